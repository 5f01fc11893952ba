// row_stats.cu -- one-read row statistics of temperature-scaled logits:
// argmax, Gumbel-max sample, softmax entropy and (optionally) the softmax in
// bf16/fp16 (page "vllm.model_executor.models.diffusion_gemma_sampler",
// module docstring, sample_row_stats and sample_row_stats_reference), and in
// the same read the top-k logprobs of the rows of converged slots
// (stash_converged_logprobs, _lp_topk_kernel).
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
//     sum" of the page); arrive on the row's first-half barrier. Division by
//     Te > 0 is monotone, so while |M_w| < 256 the warp works on the raw
//     logits: the max is found among them, only the few candidates for the
//     argmax are divided (exactly), and e = 2^(x log2(e) / Te - c) with c the
//     rounded reference is within a relative 2^-15 of e^(s - M_w). Warps
//     with larger scaled values divide every logit exactly first.
//   second half of row k-LAG, once the poller has merged the row:
//     - the probabilities e * e^(M_w - M) / S (rounded to nearest even,
//       written to HBM);
//     - the pruned race against the row's B, the best Gumbel-max score of
//       the warps' argmax elements (an element can only win if
//       1 - u <= -log u <= e^(s - B) = e * e^(M_w - B); the float4 groups
//       that pass a bound on their largest e go on a per-warp list, shared
//       out one Philox call per lane; the few survivors are rescored
//       exactly from their logits);
//     - for a converged row, the top-k candidates: the logits at or above
//       the row's threshold, rescored exactly and keyed by (value, lower
//       column) into the CTA's list. The threshold is the least, over the
//       team's G CTAs, of each CTA's r-th largest warp maximum, r =
//       ceil(k / G): G * r >= k distinct elements reach it, so the row's top
//       k all do;
//     then arrive on the row's second-half barrier, which frees the stage.
// Publisher warp: per row, combines the compute warps' first-half partials
//   into the CTA's first record (with the Gumbel-max scores of the warps'
//   argmax elements, one lane per warp, and the CTA's r-th largest raw warp
//   maximum when top-k is on) and publishes it; LAG rows later publishes the race best
//   and the CTA's top-k candidates (the k best when there are more), and
//   refills the freed stage with a later row (bulk copy), that row's
//   temperature quotient computed once for the CTA.
// Poller warp: per row, reads the team's first records (M, S, W, argmax, B,
//   the threshold candidates) and merges them for the compute warps; member 0 writes
//   argmax and entropy. For the row LAG+1 earlier it reads the race bests
//   (member 0 writes the sample) and the team's top-k candidates: every CTA
//   ranks its own candidates among all of them and writes rank r < k to
//   position r with logprob s - M - log S. A row whose candidates overflow
//   the fixed buffers (many equal values, or too few warp maxima for a
//   threshold) goes on a list that the exact top-k kernel finishes.
// LAG rows between a row's halves cover the team exchange, a round trip
// through L2. In top-k-only mode the rows of unconverged slots are skipped
// (no read, no exchange) but keep their place in the barrier protocol.
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
static_assert(kRing >= 2 * 2 + 2, "exchange ring too short for LAG 2");

// Top-k in the row kernel.
constexpr int kTopkMaxK = 64;          // larger k use the exact top-k kernel
constexpr int kTopkCtaCap = 128;       // candidates of one CTA row
constexpr int kTopkRowCap = 512;       // candidates of one team row
constexpr int kTopkRing = 4;           // CTA candidate lists, by row % 4
constexpr uint32_t kHardRow = 0xFFFFFFFFu;  // count word: candidates overflowed
constexpr int kAWords = 6;             // first record: M, S, W, argmax, B, B column
constexpr int kAWordsTopk = kAWords + 2;  // + the CTA's threshold candidate (and a pad word)
constexpr int kHardListOffset = 64;    // int32 index of the first row of the hard-row list
constexpr int kHeadKeys = 7;           // candidate keys read with a candidate record's count
constexpr int kHeadWords = 2 + 2 * kHeadKeys;

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
    uint64_t* xchg;     // exchange records, xstride words per CTA
    int* err;
    const uint8_t* keep;  // per global slot (top-k rows), or null: every row
    int32_t* out_ids;
    float* out_lp;
    int32_t* hard;        // [0]: count; rows from [kHardListOffset]
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
    int32_t stats;      // argmax / sample / entropy / probs wanted
    int32_t k;          // top-k of converged rows (0: none)
    int32_t a_words;    // words of a first record
    int32_t xstride;    // words of a CTA's exchange area
};

// Test hook state: the next launch withholds one record (see
// drs_test_inject_fault).
std::atomic<int> g_inject_fault{0};

struct WarpPartial {
    float m, s, w, xmax;
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
    float thr;        // top-k threshold (raw logit)
    int near_col;
    int arg;
    int noisy;
    int skip;         // no work (an unconverged row in top-k-only mode)
    int topk;         // top-k candidates wanted (a converged row)
};

// A row's temperature and its quotient, and whether it is worked on, set
// once by the publisher.
struct RowQuotient {
    float temp;
    float t, y;
    int mode;
    int work;
};

struct WarpRef {
    float mw;    // M_w
    float mxw;   // the raw max
    int raw;     // e taken from the raw logits
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
    WarpRef wref[kRowRing][kComputeWarps];
    int tk_count[kTopkRing];            // CTA candidate lists (top-k)
    int tk_hard[kTopkRing];
    int abort;                          // a wait ran out of time
};

// Shared memory after the stages: the Scratch, the warps' race lists, then
// (top-k only) the CTA candidate lists and the poller's merge buffer.
__host__ __device__ constexpr size_t scratch_bytes() {
    return (sizeof(Scratch) + 127) & ~static_cast<size_t>(127);
}
__host__ __device__ constexpr size_t worklist_bytes(int vec4) {
    return (static_cast<size_t>(kComputeWarps) * 32 * vec4 * sizeof(uint16_t) + 127) &
           ~static_cast<size_t>(127);
}
__host__ __device__ constexpr size_t topk_smem_bytes() {
    return static_cast<size_t>(kTopkRing) * kTopkCtaCap * 8 + static_cast<size_t>(kTopkRowCap) * 8;
}

__device__ __forceinline__ void set_comp(float4& v, int q, float x) {
    if (q == 0) v.x = x;
    else if (q == 1) v.y = x;
    else if (q == 2) v.z = x;
    else v.w = x;
}

// Two probabilities rounded to nearest even and packed (first in the low
// half): bf16 or fp16.
template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
    if (BF16) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// A thread's probabilities of one row: e * f_w for its float4 slots,
// rounded and stored (8-byte stores when the row allows them).
template <bool BF16, int VEC4>
__device__ __forceinline__ void write_probs(const float4 (&e)[VEC4], float f_w, uint16_t* prow,
                                            bool vec, int nslot4, int nfull4, int ncols, int tid) {
#pragma unroll
    for (int i = 0; i < VEC4; ++i) {
        const int f = i * kCompute + tid;
        if (i * kCompute >= nslot4 || f >= nslot4) continue;
        const uint32_t lo = pack2<BF16>(e[i].x * f_w, e[i].y * f_w);
        const uint32_t hi = pack2<BF16>(e[i].z * f_w, e[i].w * f_w);
        if (vec && f < nfull4) {
            __stcs(reinterpret_cast<uint2*>(prow + 4 * f), make_uint2(lo, hi));
        } else {
            const uint16_t code[4] = {static_cast<uint16_t>(lo), static_cast<uint16_t>(lo >> 16),
                                      static_cast<uint16_t>(hi), static_cast<uint16_t>(hi >> 16)};
            for (int q = 0; q < 4; ++q)
                if (4 * f + q < ncols) prow[4 * f + q] = code[q];
        }
    }
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

__device__ __forceinline__ int warp_sum_i(int v) {
    int r;
    asm volatile("redux.sync.add.s32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
    return r;
}

// Order-preserving unsigned form of an fp32 value (-inf lowest).
__device__ __forceinline__ uint32_t ord32(float x) {
    const uint32_t b = __float_as_uint(x);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Top-k key: value (with -0.0 as +0.0) in the high word, then the lower
// column first (the _lp_topk_kernel key order).
__device__ __forceinline__ uint64_t topk_key(float s, int col) {
    return (static_cast<uint64_t>(ord32(s + 0.0f)) << 32) |
           static_cast<uint32_t>(0x7FFFFFFF - col);
}
__device__ __forceinline__ float key_value(uint64_t key) {
    const uint32_t o = static_cast<uint32_t>(key >> 32);
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}
__device__ __forceinline__ int key_col(uint64_t key) {
    return 0x7FFFFFFF - static_cast<int>(static_cast<uint32_t>(key));
}

// Temperature of a global row: temps[row / canvas_len].
__device__ __forceinline__ uint64_t row_slot(const RowStatsParams& p, uint64_t grow_id) {
    return p.index32 ? static_cast<uint64_t>(static_cast<uint32_t>(grow_id) /
                                             static_cast<uint32_t>(p.canvas_len))
                     : grow_id / static_cast<uint64_t>(p.canvas_len);
}

// Tag of the records of a team's row sequence k (never 0: rings are zeroed
// before each launch).
__device__ __forceinline__ uint32_t record_tag(int k) { return static_cast<uint32_t>(k) + 1u; }

// A CTA's exchange area: kRing first records (a_words words each), kRing
// second records (2 words) and, with top-k, kRing candidate records
// (2 + 2k words: count, pad, then each key as two tagged halves).
__device__ __forceinline__ uint64_t* rec_a(const RowStatsParams& p, int cta, int slot) {
    return p.xchg + static_cast<size_t>(cta) * p.xstride + slot * p.a_words;
}
__device__ __forceinline__ uint64_t* rec_b(const RowStatsParams& p, int cta, int slot) {
    return p.xchg + static_cast<size_t>(cta) * p.xstride + kRing * p.a_words + slot * 2;
}
__device__ __forceinline__ uint64_t* rec_k(const RowStatsParams& p, int cta, int slot) {
    return p.xchg + static_cast<size_t>(cta) * p.xstride + kRing * (p.a_words + 2) +
           static_cast<size_t>(slot) * (2 + 2 * p.k);
}

// Poll n words (n even, 16-byte aligned) until every tag is `tag`.
template <int N>
__device__ __forceinline__ bool poll_words(const uint64_t* w, int n, uint32_t tag, uint64_t (&out)[N],
                                           uint64_t t0) {
    for (uint32_t it = 0;; ++it) {
        bool ok = true;
#pragma unroll
        for (int i = 0; i < N; i += 2) {
            if (i < n) {
                ld_relaxed_v2(w + i, out[i], out[i + 1]);
                ok &= static_cast<uint32_t>(out[i]) == tag && static_cast<uint32_t>(out[i + 1]) == tag;
            }
        }
        if (ok) return true;
        if ((it & 15u) == 15u && global_timer_ns() - t0 > kWaitLimitNs) return false;
        __nanosleep(32);
    }
}

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

__device__ __forceinline__ ScaledQuotient quotient_of(const RowQuotient& rq) {
    ScaledQuotient sq;
    sq.t = rq.t;
    sq.y = rq.y;
    sq.mode = rq.mode;
    return sq;
}

// Score the survivors `bits` of the float4 group starting at column c4
// exactly: s = x / Te from the logit in global memory (the stage holds e
// only), g from the group's Philox words; keep the best (score, column).
// The column that set the best already was scored the same way.
__device__ __noinline__ WarpBest race_rescore(uint32_t bits, const float* row_logits, int c4,
                                              uint4 w, const RowQuotient rq, int skip_col,
                                              WarpBest best) {
    const ScaledQuotient sq = quotient_of(rq);
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

// Top-k candidates of one thread: the elements of `mask` (bit 4i+q: slot
// i, component q) whose logit reaches the row's threshold, rescored exactly
// and appended to the CTA list. Returns false if the list overflowed.
__device__ __noinline__ bool topk_collect(uint64_t mask, const float* row_logits, int col0, int tid,
                                          float thr, const RowQuotient rq, int* count,
                                          uint64_t* list) {
    const ScaledQuotient sq = quotient_of(rq);
    bool ok = true;
    while (mask) {
        const int b = __ffsll(static_cast<long long>(mask)) - 1;
        mask &= mask - 1;
        const int c = col0 + 4 * ((b >> 2) * kCompute + tid) + (b & 3);
        const float x = __ldg(row_logits + c);
        if (!(x >= thr)) continue;
        const int pos = atomicAdd(count, 1);
        if (pos < kTopkCtaCap) list[pos] = topk_key(sq.exact(x), c);
        else ok = false;
    }
    return ok;
}

}  // namespace

template <int VEC4, int LAG, int NSTAGE>
__global__ void __launch_bounds__(kThreads, 1)
    row_stats_kernel(const __grid_constant__ RowStatsParams p) {
    static_assert(NSTAGE <= kMaxStages && NSTAGE >= LAG + 2, "stages");
    extern __shared__ __align__(128) unsigned char smem[];
    Scratch& sc = *reinterpret_cast<Scratch*>(smem + NSTAGE * p.stage_bytes);
    uint16_t* worklists =
        reinterpret_cast<uint16_t*>(smem + NSTAGE * p.stage_bytes + scratch_bytes());
    uint64_t* tk_lists = reinterpret_cast<uint64_t*>(smem + NSTAGE * p.stage_bytes +
                                                     scratch_bytes() + worklist_bytes(VEC4));
    uint64_t* tk_merge = tk_lists + kTopkRing * kTopkCtaCap;
    volatile int* abort_flag = &sc.abort;
    const bool use_tma = p.use_tma != 0;
    const bool stats = p.stats != 0;
    const int K = p.k;

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
    auto kept = [&](int k) { return p.keep == nullptr || p.keep[row_slot(p, grow_of(k))] != 0; };
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
        for (int r = 0; r < kTopkRing; ++r) {
            sc.tk_count[r] = 0;
            sc.tk_hard[r] = 0;
        }
        fence_barrier_init();
        sc.abort = 0;
    }
    __syncthreads();  // the only CTA barrier: everything after is mbarriers

    if (warp < kComputeWarps) {
        // ======================= compute warps ==================================
        uint16_t* list = worklists + warp * 32 * VEC4;
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
                if (rq.work) {
                    const ScaledQuotient sq = quotient_of(rq);
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
                    // exact(x) == M_w needs x >= mxw - Te * ulp(M_w), so only
                    // the slots whose max reaches that are searched, their
                    // logits read again (the stage still holds them).
                    const float cthr = mxw - fmaxf(fabsf(mxw) * 0x1p-20f, rq.t * 0x1p-140f);
                    int arg_t = INT_MAX;
                    if (stats && mt >= cthr && mw != -INFINITY) {
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
                    const int aw = stats ? warp_min_i(arg_t) : INT_MAX;

                    // t = (s - M_w) log2(e): raw domain x * log2(e)/Te - c with
                    // c = RN(mxw * log2(e)/Te), else (s - M_w) * log2(e); -inf
                    // gives a finite t whose e is 0
                    float lscale, cref;
                    if (raw) {
                        lscale = kLog2e * sq.y;
                        cref = mxw * lscale;
                    } else {
#pragma unroll
                        for (int i = 0; i < VEC4; ++i) {
                            v[i].x = sq.exact(v[i].x) - mw;
                            v[i].y = sq.exact(v[i].y) - mw;
                            v[i].z = sq.exact(v[i].z) - mw;
                            v[i].w = sq.exact(v[i].w) - mw;
                        }
                        lscale = kLog2e;
                        cref = 0.0f;
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
                        sc.p1[k & (kRowRing - 1)][warp] = WarpPartial{mw, sw, ww, mxw, aw};
                        sc.wref[k & (kRowRing - 1)][warp] = WarpRef{mw, mxw, raw ? 1 : 0};
                    }
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
                WarpBest wb{-INFINITY, INT_MAX};
                if (!ri.skip) {
                    const WarpRef wr = sc.wref[j & (kRowRing - 1)][warp];
                    const float mw = wr.mw;
                    const int64_t frow = row_of(j);
                    const float* frow_logits = p.logits + frow * p.row_stride;
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
                    if (stats && ri.noisy) {
#pragma unroll
                        for (int i = 0; i < VEC4; ++i)
                            if (max4(e[i]) * r_w >= 0x1p-24f) pmask |= 1u << i;
                    }

                    // top-k candidates: e >= e_thr is implied by x >= thr (the
                    // exponent lowered by 2^-8 for rounding); too low an e_thr
                    // leaves the row to the exact kernel.
                    uint64_t kmask = 0;
                    bool khard = false;
                    if (ri.topk) {
                        const RowQuotient rq = sc.rq[j & (kRowRing - 1)];
                        float t_thr;
                        if (ri.thr == -INFINITY) {
                            t_thr = -INFINITY;
                        } else if (wr.raw) {
                            const float lscale = kLog2e * rq.y;
                            t_thr = fmaf(ri.thr, lscale, -(wr.mxw * lscale));
                        } else {
                            t_thr = (quotient_of(rq).exact(ri.thr) - mw) * kLog2e;
                        }
                        // no threshold (fewer warp maxima than k, or the k-th
                        // is -inf): the whole row goes to the exact kernel;
                        // an all -inf warp has no candidate above a finite one
                        if (ri.thr == -INFINITY) {
                            khard = true;
                        } else if (mw != -INFINITY) {
                            if (!(t_thr - 0x1p-8f >= -120.0f)) {
                                khard = true;
                            } else {
                                const float e_thr = ex2_approx(t_thr - 0x1p-8f);
#pragma unroll
                                for (int i = 0; i < VEC4; ++i)
                                    if (max4(e[i]) >= e_thr)
#pragma unroll
                                        for (int q = 0; q < 4; ++q)
                                            if (comp(e[i], q) >= e_thr) kmask |= 1ull << (4 * i + q);
                            }
                        }
                    }

                    if (stats && p.probs_dtype != 0) {
                        // e^(s - M) / S = e * e^(M_w - M) / S; a row that is -inf
                        // everywhere gives NaN (every e is finite)
                        const float big_m = ri.row_max;
                        const float f_w = big_m == -INFINITY ? NAN
                                          : mw == -INFINITY ? 0.0f
                                                            : ex2_approx(fmaf(mw - big_m, kLog2e, -ri.log2s));
                        uint16_t* prow = static_cast<uint16_t*>(p.probs) + frow * p.probs_row_stride + col0;
                        if (p.probs_dtype == 1)
                            write_probs<true, VEC4>(e, f_w, prow, p.probs_vec != 0, nslot4, nfull4, ncols, tid);
                        else
                            write_probs<false, VEC4>(e, f_w, prow, p.probs_vec != 0, nslot4, nfull4, ncols, tid);
                    }

                    if (stats && ri.noisy) {
                        wb = WarpBest{ri.near_best, ri.near_col};
                        // the groups that pass, listed warp-wide, one per lane
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
                                wb = race_rescore(bits, frow_logits, col0 + 4 * f, w,
                                                  sc.rq[j & (kRowRing - 1)], ri.near_col, wb);
                        }
                        __syncwarp();  // the list is rewritten for the next row
                        warp_best(wb.best, wb.col);
                    }

                    if (ri.topk) {
                        bool ok = !khard;
                        if (ok && kmask)
                            ok = topk_collect(kmask, frow_logits, col0, tid, ri.thr, sc.rq[j & (kRowRing - 1)],
                                              &sc.tk_count[j & (kTopkRing - 1)],
                                              tk_lists + (j & (kTopkRing - 1)) * kTopkCtaCap);
                        if (!__all_sync(0xffffffffu, ok) && lane == 0) sc.tk_hard[j & (kTopkRing - 1)] = 1;
                    }
                }
                if (lane == 0) sc.p2[j & (kRowRing - 1)][warp] = wb;
                __syncwarp();
                if (lane == 0) mbar_arrive(&sc.b_done[j & (kRowRing - 1)]);
            }
        }
    } else if (warp == kPublisherWarp) {
        // ======================= publisher warp ==================================
        // Stage a row: its temperature quotient for the CTA, then the bulk
        // copy (or, for rows that are not 16-byte aligned, or not worked on,
        // a plain arrival: the compute warps read global memory).
        float temp_next = nrows > 0 && lane == 0 ? p.temps[row_slot(p, grow_of(0))] : 0.0f;
        auto issue_row = [&](int r) {
            if (lane == 0) {
                const float temp = temp_next;
                if (r + 1 < nrows) temp_next = p.temps[row_slot(p, grow_of(r + 1))];
                const bool work = stats || kept(r);
                const ScaledQuotient q = ScaledQuotient::of(fmaxf(temp, kTempFloor));
                sc.rq[r & (kRowRing - 1)] = RowQuotient{temp, q.t, q.y, q.mode, work ? 1 : 0};
                uint64_t* bar = &sc.full[r % NSTAGE];
                if (use_tma && work) {
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
                const RowQuotient rq = sc.rq[k & (kRowRing - 1)];
                if (rq.work) {
                    const WarpPartial wp = lane < kComputeWarps
                                               ? sc.p1[k & (kRowRing - 1)][lane]
                                               : WarpPartial{-INFINITY, 0.0f, 0.0f, -INFINITY, INT_MAX};
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
                    if (stats && rq.temp > 0.0f && wp.arg != INT_MAX) {
                        const uint4 w = noise_words_rk(p.rk, grow_of(k), static_cast<uint32_t>(wp.arg >> 2));
                        b_c = wp.m + gumbel_of_bits(word_of(w, wp.arg & 3));
                        bcol_c = wp.arg;
                    }
                    warp_best(b_c, bcol_c);
                    const bool withhold = p.fault && blockIdx.x == 0 && k == 0;
                    uint64_t* ra = rec_a(p, blockIdx.x, k & (kRing - 1));
                    const uint32_t tag = record_tag(k);
                    if (lane == 0 && !withhold) {
                        st_relaxed_v2(ra + 0, tagged(mc, tag), tagged(s_c, tag));
                        st_relaxed_v2(ra + 2, tagged(w_c, tag), tagged(static_cast<uint32_t>(a_c), tag));
                        st_relaxed_v2(ra + 4, tagged(b_c, tag), tagged(static_cast<uint32_t>(bcol_c), tag));
                    }
                    if (p.a_words > kAWords) {
                        // the r-th largest raw warp maximum of the CTA (order
                        // key), r = ceil(k / G); warps holding no column are
                        // absent (0), and fewer than r present warps give 0
                        const uint32_t o =
                            lane < kComputeWarps && lane * 32 < nslot4 ? ord32(wp.xmax) : 0u;
                        int rank = 0;  // distinct: ties go to the lower lane
#pragma unroll
                        for (int l = 0; l < kComputeWarps; ++l) {
                            const uint32_t ol = __shfl_sync(0xffffffffu, o, l);
                            rank += ol > o || (ol == o && l < lane);
                        }
                        const int r = (K + p.team - 1) / p.team;
                        const uint32_t hit = __ballot_sync(0xffffffffu, lane < kComputeWarps && rank == r - 1);
                        const uint32_t rth = hit ? __shfl_sync(0xffffffffu, o, __ffs(hit) - 1) : 0u;
                        if (lane == 0 && !withhold)
                            st_relaxed_v2(ra + kAWords, tagged(rth, tag), tagged(0u, tag));
                    }
                }
            }
            const int j = k - LAG;
            if (j >= 0) {
                // ---- second records of row j; its stage takes a later row --------
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(&sc.b_done[j & (kRowRing - 1)],
                                                               static_cast<uint32_t>((j / kRowRing) & 1)))) {
                    if (lane == 0) fail();
                    break;
                }
                const RowQuotient rq = sc.rq[j & (kRowRing - 1)];
                if (rq.work) {
                    const uint32_t tag = record_tag(j);
                    const WarpBest wb = lane < kComputeWarps ? sc.p2[j & (kRowRing - 1)][lane]
                                                             : WarpBest{-INFINITY, INT_MAX};
                    float b = wb.best;
                    int bcol = wb.col;
                    warp_best(b, bcol);
                    if (lane == 0)
                        st_relaxed_v2(rec_b(p, blockIdx.x, j & (kRing - 1)), tagged(b, tag),
                                      tagged(static_cast<uint32_t>(bcol), tag));
                    if (K > 0 && kept(j)) {
                        // the CTA's candidates: all of them, or the K best
                        const int slot = j & (kTopkRing - 1);
                        const int n = sc.tk_count[slot];
                        const bool hard = sc.tk_hard[slot] != 0 || n > kTopkCtaCap;
                        uint64_t* rk_ = rec_k(p, blockIdx.x, j & (kRing - 1));
                        const uint64_t* cl = tk_lists + slot * kTopkCtaCap;
                        int kept_n = 0;
                        if (!hard) {
                            kept_n = n < K ? n : K;
                            for (int a = lane; a < n; a += 32) {
                                const uint64_t key = cl[a];
                                int rank = 0;
                                if (n > K)
                                    for (int o = 0; o < n; ++o) rank += cl[o] > key;
                                else
                                    rank = a;
                                if (rank < K)
                                    st_relaxed_v2(rk_ + 2 + 2 * rank, tagged(static_cast<uint32_t>(key >> 32), tag),
                                                  tagged(static_cast<uint32_t>(key), tag));
                            }
                        }
                        __syncwarp();
                        if (lane == 0) {
                            st_relaxed_v2(rk_, tagged(hard ? kHardRow : static_cast<uint32_t>(kept_n), tag),
                                          tagged(0u, tag));
                            sc.tk_count[slot] = 0;
                            sc.tk_hard[slot] = 0;
                        }
                    }
                }
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
        // temperature (for the noise flag) and the keep flag are loaded a row
        // ahead.
        float temp_m = nrows > 0 ? p.temps[row_slot(p, grow_of(0))] : 0.0f;
        bool kept_m = nrows > 0 ? kept(0) : false;
        const int a_words = p.a_words;
        for (int m = 0; m < nrows + LAG + 1; ++m) {
            if (*abort_flag) break;
            const float temp = temp_m;
            const bool kept_a = kept_m;
            if (m + 1 < nrows) {
                temp_m = p.temps[row_slot(p, grow_of(m + 1))];
                kept_m = kept(m + 1);
            }
            const bool do_a = m < nrows;
            const bool work_a = do_a && (stats || kept_a);
            const int kb = m - (LAG + 1);
            const bool do_b = kb >= 0 && kb < nrows && !sc.info[kb & (kRowRing - 1)].skip;
            const bool topk_b = do_b && sc.info[kb & (kRowRing - 1)].topk;
            bool ok = true;
            uint64_t ra[kAWordsTopk], rb[2] = {0, 0}, rk8[kHeadWords];
#pragma unroll
            for (int i = 0; i < kAWordsTopk; ++i) ra[i] = 0;
#pragma unroll
            for (int i = 0; i < kHeadWords; ++i) rk8[i] = 0;
            if (do_a && !work_a) {
                // an unconverged row in top-k-only mode: no exchange, but the
                // compute warps' first half of it is awaited so that this
                // warp never runs ahead of the ring
                ok = mbar_wait_bounded(&sc.a_done[m & (kRowRing - 1)],
                                       static_cast<uint32_t>((m / kRowRing) & 1));
            }
            const bool need_b = do_b && stats;
            if (lane < p.team && (work_a || need_b || topk_b)) {
                // one polling loop over the member's first record of row m,
                // second record and candidate head (count and up to seven
                // keys) of row kb: all in flight together
                const int cta = team_id * p.team + lane;
                const uint64_t* wa = rec_a(p, cta, m & (kRing - 1));
                const uint64_t* wb2 = rec_b(p, cta, kb & (kRing - 1));
                const uint64_t* wk = rec_k(p, cta, kb & (kRing - 1));
                const uint32_t ta = record_tag(m), tb = record_tag(kb);
                bool done_a = !work_a, done_b = !need_b, done_k = !topk_b;
                const uint64_t t0 = global_timer_ns();
                for (uint32_t it = 0;; ++it) {
                    if (!done_a) {
                        bool g = true;
#pragma unroll
                        for (int i = 0; i < kAWordsTopk; i += 2)
                            if (i < a_words) {
                                ld_relaxed_v2(wa + i, ra[i], ra[i + 1]);
                                g &= static_cast<uint32_t>(ra[i]) == ta && static_cast<uint32_t>(ra[i + 1]) == ta;
                            }
                        done_a = g;
                    }
                    if (!done_b) {
                        ld_relaxed_v2(wb2, rb[0], rb[1]);
                        done_b = static_cast<uint32_t>(rb[0]) == tb && static_cast<uint32_t>(rb[1]) == tb;
                    }
                    if (!done_k) {
#pragma unroll
                        for (int i = 0; i < kHeadWords; i += 2) ld_relaxed_v2(wk + i, rk8[i], rk8[i + 1]);
                        if (static_cast<uint32_t>(rk8[0]) == tb && static_cast<uint32_t>(rk8[1]) == tb) {
                            const uint32_t c = payload_u(rk8[0]);
                            const int nk = c == kHardRow ? 0 : (c < static_cast<uint32_t>(kHeadKeys) ? static_cast<int>(c) : kHeadKeys);
                            bool g = true;
#pragma unroll
                            for (int i = 0; i < kHeadKeys; ++i)
                                if (i < nk)
                                    g &= static_cast<uint32_t>(rk8[2 + 2 * i]) == tb &&
                                         static_cast<uint32_t>(rk8[3 + 2 * i]) == tb;
                            done_k = g;
                        }
                    }
                    if (done_a && done_b && done_k) break;
                    if ((it & 15u) == 15u && global_timer_ns() - t0 > kWaitLimitNs) {
                        ok = false;
                        break;
                    }
                    __nanosleep(32);
                }
            }
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) fail();
                break;
            }
            const bool have = lane < p.team;
            if (do_a) {
                RowInfo ri{};
                ri.skip = work_a ? 0 : 1;
                if (work_a) {
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
                    ri.row_max = big_m;
                    ri.log2s = s_tot > 0.0f ? log2f(s_tot) : 0.0f;
                    ri.near_best = b_m;
                    ri.near_col = bc_m;
                    ri.arg = arg_row;
                    ri.noisy = stats && temp > 0.0f && big_m != -INFINITY;
                    ri.topk = K > 0 && kept_a;
                    ri.thr = -INFINITY;
                    if (ri.topk) {
                        // the least of the team's threshold candidates
                        const uint32_t t = warp_min_nonneg(static_cast<int>(
                            have ? payload_u(ra[kAWords]) : 0xFFFFFFFFu));
                        // absent, or below the order key of -inf: no threshold
                        if (t > 0x007FFFFFu)
                            ri.thr = __uint_as_float((t & 0x80000000u) ? (t & 0x7FFFFFFFu) : ~t);
                    }
                    if (lane == 0 && member == 0 && stats) {
                        p.argmax[frow] = arg_row;
                        p.entropy[frow] = s_tot > 0.0f ? logf(s_tot) - w_tot / s_tot : 0.0f;
                        if (!ri.noisy) p.sample[frow] = arg_row;
                    }
                }
                if (lane == 0) {
                    sc.info[m & (kRowRing - 1)] = ri;
                    mbar_arrive(&sc.info_ready[m & (kRowRing - 1)]);
                }
            }
            if (do_b) {
                const RowInfo ri = sc.info[kb & (kRowRing - 1)];
                if (stats) {
                    float b = have ? payload_f(rb[0]) : -INFINITY;
                    int bcol = have ? static_cast<int>(payload_u(rb[1])) : INT_MAX;
                    warp_best(b, bcol);
                    if (lane == 0 && ri.noisy && member == 0) {
                        float bb = ri.near_best;
                        int bbc = ri.near_col;
                        if (beats(b, bcol, bb, bbc)) {
                            bb = b;
                            bbc = bcol;
                        }
                        p.sample[row_of(kb)] = bb != -INFINITY ? bbc : ri.arg;
                    }
                }
                if (topk_b) {
                    // the team's candidates: counts first, then the keys into
                    // the merge buffer at each member's offset
                    const uint32_t tag = record_tag(kb);
                    bool okk = true;
                    const uint32_t cnt = have ? payload_u(rk8[0]) : 0u;
                    const bool any_hard = __any_sync(0xffffffffu, cnt == kHardRow);
                    const int c = any_hard ? 0 : static_cast<int>(cnt);
                    const int total = warp_sum_i(c);
                    int off = c;  // inclusive scan
#pragma unroll
                    for (int d = 1; d < 32; d <<= 1) {
                        const int y = __shfl_up_sync(0xffffffffu, off, d);
                        if (lane >= d) off += y;
                    }
                    off -= c;
                    const int own_off = __shfl_sync(0xffffffffu, off, member);
                    const int own_n = __shfl_sync(0xffffffffu, c, member);
                    if (any_hard || total > kTopkRowCap || total < K) {
                        if (lane == 0 && member == 0) {
                            const int idx = atomicAdd(p.hard, 1);
                            p.hard[kHardListOffset + idx] = static_cast<int32_t>(row_of(kb));
                        }
                    } else {
                        if (have && c > 0) {
                            // the first keys came with the head; the rest are
                            // read four at a time
#pragma unroll
                            for (int r = 0; r < kHeadKeys; ++r)
                                if (r < c)
                                    tk_merge[off + r] = (static_cast<uint64_t>(payload_u(rk8[2 + 2 * r])) << 32) |
                                                        payload_u(rk8[3 + 2 * r]);
                            const uint64_t* src = rec_k(p, team_id * p.team + lane, kb & (kRing - 1)) + 2;
                            const uint64_t t0 = global_timer_ns();
                            for (int r0 = kHeadKeys; r0 < c && okk; r0 += 4) {
                                uint64_t kw[8];
                                const int nw = 2 * (c - r0 < 4 ? c - r0 : 4);
                                okk = poll_words(src + 2 * r0, nw, tag, kw, t0);
#pragma unroll
                                for (int r = 0; r < 4; ++r)
                                    if (2 * r < nw)
                                        tk_merge[off + r0 + r] =
                                            (static_cast<uint64_t>(payload_u(kw[2 * r])) << 32) | payload_u(kw[2 * r + 1]);
                            }
                        }
                        if (!__all_sync(0xffffffffu, okk)) {
                            if (lane == 0) fail();
                            break;
                        }
                        __syncwarp();
                        // rank this CTA's candidates among the team's, one
                        // candidate at a time, the count spread over the lanes
                        const int64_t frow = row_of(kb);
                        const float lns = ri.log2s * kLn2;
                        for (int a = 0; a < own_n; ++a) {
                            const uint64_t key = tk_merge[own_off + a];
                            int cnt = 0;
                            for (int o = lane; o < total; o += 32) cnt += tk_merge[o] > key;
                            const int rank = warp_sum_i(cnt);
                            if (lane == 0 && rank < K) {
                                const float sv = key_value(key);
                                p.out_ids[frow * K + rank] = key_col(key);
                                p.out_lp[frow * K + rank] =
                                    ri.row_max == -INFINITY ? NAN : (sv - ri.row_max) - lns;
                            }
                        }
                        __syncwarp();  // the buffer is refilled for the next row
                    }
                }
            }
        }
    }
}

}  // namespace drs

namespace drs {
namespace {

struct RowStatsPlan {
    RowPlan rows;
    int lag;     // 2 or 1
    int nstage;  // 5 (LAG 2), 4 or 3 (LAG 1)
    int vec4;    // float4 slots per compute thread
};

size_t fixed_smem(int vec4, bool topk) {
    return scratch_bytes() + worklist_bytes(vec4) + (topk ? topk_smem_bytes() : 0);
}

// Team size G for one CTA per SM with 448 compute threads. The chunk must
// fit the registers and the stages shared memory. An iteration costs about
// max(chunk, round trip / LAG) + 1500 columns of work, the round trip of the
// team exchange through L2 (about 2.6 us) being worth some 18000 columns;
// the plan minimises ceil(rows / teams) times that, with teams = min(rows,
// sms / G) and the three-stage form counted 25% dearer. Ties go to the
// earlier form, then the smaller G.
RowStatsPlan plan_row_stats(int64_t rows, int vocab, int sms, bool topk) {
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
        const size_t budget = kSmemPerCta - fixed_smem(fm.vec4, topk);
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
drs_status launch_form(RowStatsParams& prm, int grid, size_t smem, cudaStream_t stream) {
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

// Words of a CTA's exchange area.
size_t xchg_words(int32_t k) {
    const size_t a = k > 0 ? kAWordsTopk : kAWords;
    return kRing * (a + 2) + (k > 0 ? kRing * (2 + 2 * static_cast<size_t>(k)) : 0);
}
size_t round_up(size_t n, size_t a) { return (n + a - 1) / a * a; }
size_t hard_list_bytes(int64_t rows) {
    return round_up(4 * (static_cast<size_t>(kHardListOffset) + static_cast<size_t>(rows)), kWorkspaceAlign);
}
size_t xchg_bytes(int32_t k) { return round_up(1024 * xchg_words(k) * 8, kWorkspaceAlign); }

drs_status run_rows(const RowCall& c, void* xchg, int32_t* hard, cudaStream_t stream) {
    const int sms = sm_count();
    if (sms <= 0) return DRS_ERR_CUDA;
    const bool topk = c.k > 0;
    const RowStatsPlan rsp = plan_row_stats(c.rows, static_cast<int>(c.vocab), sms, topk);
    const RowPlan& plan = rsp.rows;
    if (!plan.team) return DRS_ERR_UNSUPPORTED;
    // per-team row counts are int
    if ((c.rows + plan.num_teams - 1) / plan.num_teams > INT_MAX / 2) return DRS_ERR_UNSUPPORTED;

    RowStatsParams prm{};
    prm.logits = c.logits;
    prm.row_stride = c.row_stride;
    prm.rows = c.rows;
    prm.row0 = c.row0;
    prm.temps = c.temps;
    prm.canvas_len = c.canvas_len;
    prm.argmax = c.argmax;
    prm.sample = c.sample;
    prm.entropy = c.entropy;
    prm.probs = c.probs;
    prm.probs_row_stride = c.probs_row_stride;
    prm.xchg = static_cast<uint64_t*>(xchg);
    prm.err = device_error_flag();
    prm.keep = c.keep;
    prm.out_ids = c.out_ids;
    prm.out_lp = c.out_lp;
    prm.hard = hard;
    prm.rk = PhiloxRoundKeys::of(c.seed);
    prm.vocab = static_cast<int32_t>(c.vocab);
    prm.team = plan.team;
    prm.chunk = plan.chunk;
    prm.num_teams = plan.num_teams;
    prm.probs_dtype = static_cast<int32_t>(c.probs_dtype);
    prm.probs_vec = c.probs && aligned(c.probs, 8) && (c.probs_row_stride % 4 == 0);
    prm.index32 = (c.row0 + c.rows <= static_cast<int64_t>(UINT32_MAX)) &&
                  (c.canvas_len <= static_cast<int64_t>(UINT32_MAX));
    prm.fault = g_inject_fault.exchange(0);
    prm.stats = c.stats ? 1 : 0;
    prm.k = c.k;
    prm.a_words = topk ? kAWordsTopk : kAWords;
    prm.xstride = static_cast<int32_t>(xchg_words(c.k));
    if (!prm.err) return DRS_ERR_CUDA;

    // Shared memory: the stages of one chunk each (filled by bulk copies when
    // rows start 16-byte aligned; in every case they keep a row's e until its
    // second half), the scratch, the race lists, the top-k buffers.
    const bool tma = aligned(c.logits, 16) && (c.row_stride % 4 == 0);
    prm.stage_bytes = (plan.chunk * 4 + 127) & ~127;
    prm.use_tma = tma ? 1 : 0;
    const size_t smem =
        static_cast<size_t>(rsp.nstage) * prm.stage_bytes + fixed_smem(rsp.vec4, topk);
    if (smem > kSmemPerCta) return DRS_ERR_UNSUPPORTED;
    const int grid = plan.team * plan.num_teams;
    // Zero the records this launch uses (a zero tag matches no row) and the
    // count of the hard-row list.
    if (cudaMemsetAsync(xchg, 0, static_cast<size_t>(grid) * xchg_words(c.k) * 8, stream) != cudaSuccess)
        return DRS_ERR_CUDA;
    if (hard && cudaMemsetAsync(hard, 0, 4, stream) != cudaSuccess) return DRS_ERR_CUDA;
    if (rsp.lag == 2) return launch_form<kVec4Lag2, 2, 5>(prm, grid, smem, stream);
    if (rsp.nstage == 4) return launch_form<kVec4Lag1, 1, 4>(prm, grid, smem, stream);
    return launch_form<kVec4Lag1, 1, 3>(prm, grid, smem, stream);
}

drs_status check_stats_args(const float* logits, int64_t rows, int64_t vocab, int64_t row_stride,
                            const float* temps, int64_t canvas_len, int64_t row0, int64_t* argmax,
                            int64_t* sample, float* entropy, drs_probs_dtype probs_dtype,
                            void* probs, int64_t probs_row_stride) {
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
    return DRS_OK;
}

// Top-k of the converged rows into a workspace laid out as: the split
// kernels' workspace (the hard-row list first), the exact kernel's records.
drs_status run_topk(RowCall c, void* workspace, cudaStream_t stream) {
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    const int32_t* hard = reinterpret_cast<const int32_t*>(ws);
    void* exact_ws = ws + split_workspace_bytes(c.rows, c.vocab, c.k > split_max_k() ? 0 : c.k);
    if (c.k > split_max_k()) {
        // larger k: the row statistics alone, then the exact kernel on every
        // converged row
        if (c.stats) {
            RowCall s = c;
            s.k = 0;
            s.keep = nullptr;
            const drs_status st = split_rows(s, workspace, stream);
            if (st != DRS_OK) return st;
        }
        return exact_topk(c.logits, c.rows, c.vocab, c.row_stride, c.row0, c.temps, c.canvas_len,
                          c.keep, nullptr, c.k, c.out_ids, c.out_lp, exact_ws, stream);
    }
    const drs_status st = split_rows(c, workspace, stream);
    if (st != DRS_OK) return st;
    // the rows the split kernels left (no threshold, or too many candidates)
    return exact_topk(c.logits, c.rows, c.vocab, c.row_stride, c.row0, c.temps, c.canvas_len,
                      c.keep, hard, c.k, c.out_ids, c.out_lp, exact_ws, stream);
}

}  // namespace
}  // namespace drs

int drs::take_injected_fault() { return drs::g_inject_fault.exchange(0); }

extern "C" void drs_test_inject_fault(int code) { drs::g_inject_fault.store(code); }

extern "C" size_t drs_row_stats_workspace_bytes(int64_t rows, int64_t vocab) {
    if (rows < 0 || vocab < 1) return 0;
    return drs::split_workspace_bytes(rows, vocab, 0);
}

extern "C" drs_status drs_row_stats(const float* logits, int64_t rows, int64_t vocab,
                                    int64_t row_stride, const float* temps,
                                    int64_t canvas_len, uint64_t seed, int64_t row0,
                                    int64_t* argmax, int64_t* sample, float* entropy,
                                    drs_probs_dtype probs_dtype, void* probs,
                                    int64_t probs_row_stride, void* workspace,
                                    size_t workspace_bytes, void* stream) {
    using namespace drs;
    const drs_status chk = check_stats_args(logits, rows, vocab, row_stride, temps, canvas_len,
                                            row0, argmax, sample, entropy, probs_dtype, probs,
                                            probs_row_stride);
    if (chk != DRS_OK) return chk;
    if (rows == 0) return DRS_OK;
    const size_t need = drs_row_stats_workspace_bytes(rows, vocab);
    if (!workspace || workspace_bytes < need || !aligned(workspace, kWorkspaceAlign))
        return DRS_ERR_INVALID_ARG;
    RowCall c{logits, rows, vocab, row_stride, temps, canvas_len, seed, row0, argmax, sample,
              entropy, probs_dtype, probs, probs_row_stride, nullptr, 0, nullptr, nullptr, true};
    return split_rows(c, workspace, static_cast<cudaStream_t>(stream));
}

extern "C" size_t drs_row_stats_topk_workspace_bytes(int64_t rows, int64_t vocab, int32_t k) {
    if (k <= 0 || rows < 0 || vocab < 1) return 0;
    const int32_t ks = k > drs::split_max_k() ? 0 : k;
    return drs::split_workspace_bytes(rows, vocab, ks) + drs::exact_topk_workspace_bytes(k);
}

extern "C" drs_status drs_row_stats_topk(const float* logits, int64_t rows, int64_t vocab,
                                         int64_t row_stride, const float* temps,
                                         int64_t canvas_len, uint64_t seed, int64_t row0,
                                         int64_t* argmax, int64_t* sample, float* entropy,
                                         drs_probs_dtype probs_dtype, void* probs,
                                         int64_t probs_row_stride, const uint8_t* keep, int32_t k,
                                         int32_t* out_ids, float* out_logprobs, void* workspace,
                                         size_t workspace_bytes, void* stream) {
    using namespace drs;
    const drs_status chk = check_stats_args(logits, rows, vocab, row_stride, temps, canvas_len,
                                            row0, argmax, sample, entropy, probs_dtype, probs,
                                            probs_row_stride);
    if (chk != DRS_OK) return chk;
    if (k < 0 || k > vocab || k > exact_topk_max_k()) return DRS_ERR_INVALID_ARG;
    if (k > 0 && (!keep || !out_ids || !out_logprobs)) return DRS_ERR_INVALID_ARG;
    if (rows == 0) return DRS_OK;
    if (k == 0)
        return drs_row_stats(logits, rows, vocab, row_stride, temps, canvas_len, seed, row0,
                             argmax, sample, entropy, probs_dtype, probs, probs_row_stride,
                             workspace, workspace_bytes, stream);
    const size_t need = drs_row_stats_topk_workspace_bytes(rows, vocab, k);
    if (!workspace || workspace_bytes < need || !aligned(workspace, kWorkspaceAlign))
        return DRS_ERR_INVALID_ARG;
    RowCall c{logits, rows, vocab, row_stride, temps, canvas_len, seed, row0, argmax, sample,
              entropy, probs_dtype, probs, probs_row_stride, keep, k, out_ids, out_logprobs, true};
    return run_topk(c, workspace, static_cast<cudaStream_t>(stream));
}

extern "C" size_t drs_topk_workspace_bytes(int64_t rows, int64_t vocab, int32_t k) {
    return drs_row_stats_topk_workspace_bytes(rows, vocab, k);
}

extern "C" drs_status drs_topk_logprobs(const float* logits, int64_t rows, int64_t vocab,
                                        int64_t row_stride, const float* temps,
                                        int64_t canvas_len, const uint8_t* keep, int32_t k,
                                        int32_t* out_ids, float* out_logprobs, void* workspace,
                                        size_t workspace_bytes, void* stream) {
    using namespace drs;
    if (rows < 0 || canvas_len < 1 || k < 0) return DRS_ERR_INVALID_ARG;
    if (vocab < 1 || row_stride < vocab) return DRS_ERR_INVALID_ARG;
    if (vocab > DRS_MAX_VOCAB) return DRS_ERR_UNSUPPORTED;
    if (k > vocab || k > exact_topk_max_k()) return DRS_ERR_INVALID_ARG;
    if (rows % canvas_len != 0) return DRS_ERR_INVALID_ARG;
    if (k == 0 || rows == 0) return DRS_OK;
    if (!logits || !temps || !keep || !out_ids || !out_logprobs) return DRS_ERR_INVALID_ARG;
    if (!aligned(logits, 4)) return DRS_ERR_INVALID_ARG;
    const size_t need = drs_topk_workspace_bytes(rows, vocab, k);
    if (!workspace || workspace_bytes < need || !aligned(workspace, kWorkspaceAlign))
        return DRS_ERR_INVALID_ARG;
    RowCall c{logits, rows, vocab, row_stride, temps, canvas_len, 0, 0, nullptr, nullptr,
              nullptr, DRS_PROBS_NONE, nullptr, 0, keep, k, out_ids, out_logprobs, false};
    return run_topk(c, workspace, static_cast<cudaStream_t>(stream));
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

constexpr size_t kNoallocWorkspaceBytes = static_cast<size_t>(640) * 1024;
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
    const drs_status chk = drs::check_stats_args(logits, rows, vocab, row_stride, temps,
                                                 canvas_len, row0, argmax, sample, entropy,
                                                 probs_dtype, probs, probs_row_stride);
    if (chk != DRS_OK) return chk;
    if (rows == 0) return DRS_OK;
    // rows in batches whose workspace fits the array (one row always does)
    int64_t batch = rows;
    while (batch > 1 && drs_row_stats_workspace_bytes(batch, vocab) > kNoallocWorkspaceBytes)
        batch = (batch + 1) / 2;
    if (drs_row_stats_workspace_bytes(batch, vocab) > kNoallocWorkspaceBytes)
        return DRS_ERR_UNSUPPORTED;
    drs_status st = DRS_OK;
    void* ws = noalloc_workspace(&st);
    if (!ws) return st;
    const size_t pbytes = probs_dtype == DRS_PROBS_NONE ? 0 : 2;
    for (int64_t r = 0; r < rows; r += batch) {
        const int64_t n = rows - r < batch ? rows - r : batch;
        void* pr = probs ? static_cast<unsigned char*>(probs) +
                               static_cast<size_t>(r) * static_cast<size_t>(probs_row_stride) * pbytes
                         : nullptr;
        st = drs_row_stats(logits + r * row_stride, n, vocab, row_stride, temps, canvas_len, seed,
                           row0 + r, argmax + r, sample + r, entropy + r, probs_dtype, pr,
                           probs_row_stride, ws, kNoallocWorkspaceBytes, stream);
        if (st != DRS_OK) return st;
    }
    return DRS_OK;
}
