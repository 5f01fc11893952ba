// topk.cu -- top-k logprobs of the rows of converged slots (page
// "vllm.model_executor.models.diffusion_gemma_sampler": the
// stash_converged_logprobs docstring and _lp_topk_kernel).
//
// A key orders by value, then by lower column: the high word is the fp32
// bit pattern mapped to an order-preserving int32 (b ^ ((b >> 31) &
// 0x7FFFFFFF)), the low word 0x7FFFFFFF - column. Keys are distinct, so the
// top-k under them is unique. -0.0 is canonicalised to +0.0 first.
//
// Work layout: a team of G CTAs owns the G column chunks of each row (one
// CTA per SM, all resident, so their bounded waits on each other cannot
// deadlock); teams take rows round robin. Rows of slots whose keep flag is 0
// are skipped by the whole team (nothing is read or written for them). Per
// kept row, each CTA
//   1. stages its chunk (bulk copy), scales it (IEEE division by
//      max(T, 1e-10)) and computes its max m and S = sum e^(s - m);
//   2. takes as threshold the k-th largest of its 512 per-thread maximum
//      keys: those k maxima are k distinct elements at or above it, so every
//      element of the CTA's top-k is too (the block-max argument of
//      _lp_topk_kernel, with one block per thread);
//   3. ranks the candidates at or above the threshold by counting and keeps
//      the first k (if tied values make the candidates too many, an exact
//      bitwise search for the k-th largest key replaces the threshold);
//   4. publishes (m, S, its k keys) in the workspace; every CTA of the team
//      then ranks its own keys against all G*k published keys and writes
//      those of global rank r < k to position r, with logprob
//      s - M - log(sum_c S_c e^(m_c - M)).
#include <algorithm>
#include <cfloat>
#include <climits>

#include "drs_device.cuh"
#include "drs_internal.h"

namespace drs {

namespace {

constexpr int kMaxStages = 3;
constexpr int kMaxK = 2 * kThreads;  // two keys per thread in the merge
constexpr int kCandCap = 2048;    // shared-memory candidate slots
constexpr int kFastCands = 512;   // above this many, use the exact search

struct TopkParams {
    const float* logits;
    int64_t row_stride;
    int64_t rows;
    int64_t row0;             // global index of row 0 (temperature and keep slot)
    const int32_t* row_list;  // null, or [0] the count and the rows from [64]
    // With a map, the listed "rows" are entries e: logits row map_row[e],
    // temperature map_temp[e], outputs at e (the stash's rows).
    const int32_t* map_row;
    const float* map_temp;
    float* out_m;             // null, or per output row: the max scaled logit
    float* out_logs;          // and the log of the sum of e^(s - max)
    const float* temps;
    int64_t canvas_len;
    const uint8_t* keep;
    int32_t* out_ids;
    float* out_lp;
    unsigned char* xchg;
    int* err;
    uint32_t generation;
    int32_t k;
    int32_t vocab;
    int32_t team;
    int32_t chunk;
    int32_t num_teams;
    int32_t nstage;
    int32_t stage_bytes;
    int32_t rec_bytes;
    int32_t vec;              // the one-CTA kernel: rows start 16-byte aligned (float4 loads)
};

// Record header; the k keys follow it.
struct alignas(32) TopkHeader {
    uint64_t tag;
    float m;
    float s;
    int32_t count;
    int32_t pad[3];
};
static_assert(sizeof(TopkHeader) == 32, "header layout");

struct TopkScratch {
    uint64_t full[kMaxStages];
    float wmax[kWarps];
    float ws[kWarps];
    int wcnt[kWarps];
    unsigned long long wcnt64[kWarps];
    int ncand;
    int status;
    float row_max;
    float row_logs;
};

__device__ __forceinline__ void set_comp(float4& v, int q, float x) {
    if (q == 0) v.x = x;
    else if (q == 1) v.y = x;
    else if (q == 2) v.z = x;
    else v.w = x;
}

__device__ __forceinline__ int32_t key32_of(float s) {
    const int32_t b = __float_as_int(s);
    return b ^ ((b >> 31) & 0x7FFFFFFF);
}

__device__ __forceinline__ float value_of_key32(int32_t k) {
    const int32_t b = k ^ ((k >> 31) & 0x7FFFFFFF);
    return __int_as_float(b);
}

__device__ __forceinline__ int64_t make_key(float s, int col) {
    return (static_cast<int64_t>(key32_of(s)) << 32) |
           static_cast<int64_t>(0x7FFFFFFF - col);
}

constexpr int64_t kNoKey = INT64_MIN;

__device__ __forceinline__ int block_sum_int(int v, int* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    int r = (threadIdx.x & 31) < kWarps ? red[threadIdx.x & 31] : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
    __syncthreads();
    return r;
}

__device__ __forceinline__ uint32_t block_min_u32(uint32_t v, int* red) {
    asm("redux.sync.min.u32 %0, %1, 0xffffffff;" : "=r"(v) : "r"(v));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = static_cast<int>(v);
    __syncthreads();
    uint32_t r = (threadIdx.x & 31) < kWarps ? static_cast<uint32_t>(red[threadIdx.x & 31]) : 0xFFFFFFFFu;
    asm("redux.sync.min.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(r));
    __syncthreads();
    return r;
}

// The sum of v over the threads before this one (thread order), every thread.
__device__ __forceinline__ int block_excl_scan(int v, int* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += y;
    }
    if (lane == 31) red[warp] = incl;
    __syncthreads();
    int before = 0;
    for (int w = 0; w < warp; ++w) before += red[w];
    __syncthreads();
    return before + incl - v;
}

}  // namespace

template <int VEC4>
__global__ void __launch_bounds__(kThreads, 1)
    topk_kernel(const __grid_constant__ TopkParams p) {
    // a programmatic dependent launched after this kernel (the stash's
    // write) may start now: it waits for this grid before reading its results
    asm volatile("griddepcontrol.launch_dependents;");
    extern __shared__ __align__(128) unsigned char smem[];
    TopkScratch& sc = *reinterpret_cast<TopkScratch*>(smem + p.nstage * p.stage_bytes);
    int64_t* cand = reinterpret_cast<int64_t*>(
        smem + p.nstage * p.stage_bytes + ((sizeof(TopkScratch) + 127) & ~size_t(127)));

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int team_id = blockIdx.x / p.team;
    const int member = blockIdx.x - team_id * p.team;
    const int col0 = member * p.chunk;
    const int ncols = min(p.vocab - col0, p.chunk);
    const int nfull4 = ncols >> 2;
    const uint32_t copy_bytes = static_cast<uint32_t>(nfull4) * 16u;
    // the rows: every row of the call (those of unconverged slots skipped),
    // or the rows of a list whose length a previous kernel left on the device
    const int64_t nlisted = p.row_list ? static_cast<int64_t>(p.row_list[0]) : p.rows;
    const int64_t nrows = team_id < nlisted ? (nlisted - 1 - team_id) / p.num_teams + 1 : 0;
    const int K = p.k;
    const bool use_tma = p.nstage > 0;

    auto row_of = [&](int64_t j) {
        const int64_t r = team_id + j * p.num_teams;
        return p.row_list ? static_cast<int64_t>(p.row_list[64 + r]) : r;
    };
    auto logits_row = [&](int64_t r) { return p.map_row ? static_cast<int64_t>(p.map_row[r]) : r; };
    auto kept = [&](int64_t j) {
        return p.row_list != nullptr || p.keep[(p.row0 + row_of(j)) / p.canvas_len] != 0;
    };
    auto next_kept = [&](int64_t j) {
        while (j < nrows && !kept(j)) ++j;
        return j;
    };

    if (use_tma && tid == 0) {
        for (int s = 0; s < p.nstage; ++s) mbar_init(&sc.full[s], 1);
        fence_barrier_init();
    }
    __syncthreads();

    // Producer state (thread 0): next team row to stage and kept rows issued.
    int64_t issue_j = 0, issued = 0;
    auto issue_next = [&]() {
        issue_j = next_kept(issue_j);
        if (issue_j >= nrows) return false;
        const int s = static_cast<int>(issued % p.nstage);
        mbar_arrive_expect_tx(&sc.full[s], copy_bytes);
        if (copy_bytes)
            tma_load_1d(smem + s * p.stage_bytes,
                        p.logits + logits_row(row_of(issue_j)) * p.row_stride + col0, copy_bytes,
                        &sc.full[s]);
        ++issue_j;
        ++issued;
        return true;
    };
    if (use_tma && tid == 0) {
        for (int s = 0; s < p.nstage; ++s)
            if (!issue_next()) break;
    }

    bool aborted = false;
    int64_t consumed = 0;
    int64_t j = next_kept(0);
    for (int64_t kk = 0; j < nrows; ++kk, j = next_kept(j + 1)) {
        const int64_t row = row_of(j);
        const float* grow = p.logits + logits_row(row) * p.row_stride + col0;

        // ---- load and scale ------------------------------------------------
        bool timed_out = false;
        const int s = use_tma ? static_cast<int>(kk % p.nstage) : 0;
        if (use_tma)
            timed_out = !mbar_wait_bounded(&sc.full[s], static_cast<uint32_t>((kk / p.nstage) & 1));
        const float4* stage4 = reinterpret_cast<const float4*>(smem + s * p.stage_bytes);
        float4 v[VEC4];
#pragma unroll
        for (int i = 0; i < VEC4; ++i) {
            const int f = i * kThreads + tid;
            float4 x = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
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
            v[i] = x;
        }
        if (__syncthreads_or(timed_out)) {
            aborted = true;
            break;
        }
        consumed = kk + 1;
        if (use_tma && tid == 0) {
            fence_proxy_async_smem();
            issue_next();
        }
        const float temp = p.map_temp ? p.map_temp[row] : p.temps[(p.row0 + row) / p.canvas_len];
        const ScaledQuotient sq = ScaledQuotient::of(fmaxf(temp, kTempFloor));
#pragma unroll
        for (int i = 0; i < VEC4; ++i) {
            // x / te exactly (infinities kept), then -0.0 -> +0.0 (one value
            // for the order)
            v[i].x = sq.exact(v[i].x) + 0.0f;
            v[i].y = sq.exact(v[i].y) + 0.0f;
            v[i].z = sq.exact(v[i].z) + 0.0f;
            v[i].w = sq.exact(v[i].w) + 0.0f;
        }
        auto valid = [&](int i, int q) { return 4 * (i * kThreads + tid) + q < ncols; };
        auto col_of = [&](int i, int q) { return col0 + 4 * (i * kThreads + tid) + q; };

        // ---- CTA max and sum -------------------------------------------------
        float mt = -INFINITY;
        uint32_t tmax = 0;  // thread max key32, sign-flipped to unsigned order
        int nvalid = 0;
#pragma unroll
        for (int i = 0; i < VEC4; ++i)
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (valid(i, q)) {
                    const float x = comp(v[i], q);
                    mt = fmaxf(mt, x);
                    tmax = max(tmax, static_cast<uint32_t>(key32_of(x)) ^ 0x80000000u);
                    ++nvalid;
                }
        {
            const float wm = warp_max(mt);
            if (lane == 0) sc.wmax[warp] = wm;
        }
        __syncthreads();
        const float mc = warp_max(lane < kWarps ? sc.wmax[lane] : -INFINITY);
        float st = 0.0f;
        if (mc != -INFINITY) {
#pragma unroll
            for (int i = 0; i < VEC4; ++i)
#pragma unroll
                for (int q = 0; q < 4; ++q) st += ex2_approx((comp(v[i], q) - mc) * kLog2e);
        }
        {
            const float ws = warp_sum_f(st);
            if (lane == 0) sc.ws[warp] = ws;
        }

        // ---- threshold: k-th largest thread maximum --------------------------
        // Bitwise search for the largest t with #{threads: tmax >= t} >= K.
        // Threads without valid columns hold 0 and never count.
        uint32_t t = 0;
        for (int b = 31; b >= 0; --b) {
            const uint32_t c = t | (1u << b);
            if (__syncthreads_count(nvalid > 0 && tmax >= c) >= K) t = c;
        }
        // Candidates: valid elements whose key32 (unsigned order) >= t.
        if (tid == 0) sc.ncand = 0;
        __syncthreads();
#pragma unroll
        for (int i = 0; i < VEC4; ++i)
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (valid(i, q)) {
                    const float x = comp(v[i], q);
                    if ((static_cast<uint32_t>(key32_of(x)) ^ 0x80000000u) >= t) {
                        const int pos = atomicAdd(&sc.ncand, 1);
                        if (pos < kCandCap) cand[pos] = make_key(x, col_of(i, q));
                    }
                }
        __syncthreads();
        int ncand = sc.ncand;

        if (ncand > kFastCands) {
            // Tied values make the candidates too many. Exactly the CTA's
            // top `want` keys instead: t2, the want-th largest value (key32),
            // then all elements above it and the lowest columns among those
            // equal to it (keys order equal values by lower column).
            auto u32 = [&](float x) { return static_cast<uint32_t>(key32_of(x)) ^ 0x80000000u; };
            const int want = min(K, block_sum_int(nvalid, sc.wcnt));
            // the smallest candidate value is t2 when fewer than `want`
            // elements exceed it (constant rows, rows of -inf ties);
            // otherwise a bitwise search over the values
            uint32_t mn = 0xFFFFFFFFu;
#pragma unroll
            for (int i = 0; i < VEC4; ++i)
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (valid(i, q) && u32(comp(v[i], q)) >= t) mn = min(mn, u32(comp(v[i], q)));
            mn = block_min_u32(mn, sc.wcnt);
            auto count_above = [&](uint32_t c) {  // elements with value > c, block-wide
                int cnt = 0;
#pragma unroll
                for (int i = 0; i < VEC4; ++i)
#pragma unroll
                    for (int q = 0; q < 4; ++q) cnt += valid(i, q) && u32(comp(v[i], q)) > c;
                return block_sum_int(cnt, sc.wcnt);
            };
            uint32_t t2 = mn;
            int gt = count_above(mn);
            if (gt >= want) {
                // the largest c with #(value >= c) >= want
                t2 = 0;
                for (int b = 31; b >= 0; --b) {
                    const uint32_t c = t2 | (1u << b);
                    // #(value >= c) = #(value > c - 1)
                    if (count_above(c - 1) >= want) t2 = c;
                }
                gt = count_above(t2);
            }
            const int r = want - gt;  // ties at t2 to take, lowest columns first
            // the slot holding the r-th tie in column order (slot i of the
            // block covers columns [4 i kThreads, 4 (i + 1) kThreads) of the
            // chunk), then the ties before each thread within it
            int ties[VEC4];
#pragma unroll
            for (int i = 0; i < VEC4; ++i) {
                ties[i] = 0;
#pragma unroll
                for (int q = 0; q < 4; ++q) ties[i] += valid(i, q) && u32(comp(v[i], q)) == t2;
            }
            int before = 0, istar = VEC4;
#pragma unroll
            for (int i = 0; i < VEC4; ++i) {
                const int tot = block_sum_int(ties[i], sc.wcnt);
                if (istar == VEC4) {
                    if (before + tot >= r) istar = i;
                    else before += tot;
                }
            }
            int mine = 0;
#pragma unroll
            for (int i = 0; i < VEC4; ++i)
                if (i == istar) mine = ties[i];
            const int ex = block_excl_scan(mine, sc.wcnt);
            const int need = r - before;  // ties to take inside slot istar
            if (tid == 0) sc.ncand = 0;
            __syncthreads();
#pragma unroll
            for (int i = 0; i < VEC4; ++i) {
                int seen = 0;  // this thread's earlier ties in slot i
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (valid(i, q)) {
                        const float x = comp(v[i], q);
                        const uint32_t u = u32(x);
                        bool take = u > t2;
                        if (u == t2) {
                            take = i < istar || (i == istar && ex + seen < need);
                            ++seen;
                        }
                        if (take) {
                            const int pos = atomicAdd(&sc.ncand, 1);
                            if (pos < kCandCap) cand[pos] = make_key(x, col_of(i, q));
                        }
                    }
            }
            __syncthreads();
            ncand = sc.ncand;
        }

        // ---- local top-k by counting ranks ------------------------------------
        const int slot = static_cast<int>(kk % kRing);
        unsigned char* my_rec = p.xchg + (static_cast<size_t>(blockIdx.x) * kRing + slot) * p.rec_bytes;
        int64_t* my_keys = reinterpret_cast<int64_t*>(my_rec + sizeof(TopkHeader));
        const int nlocal = min(K, ncand);
        for (int c = tid; c < ncand; c += kThreads) {
            const int64_t key = cand[c];
            int rank = 0;
            for (int o = 0; o < ncand; ++o) rank += cand[o] > key;
            if (rank < nlocal) my_keys[rank] = key;
        }
        for (int c = nlocal + tid; c < K; c += kThreads) my_keys[c] = kNoKey;
        const float s_cta = warp_sum_f(lane < kWarps ? sc.ws[lane] : 0.0f);
        __syncthreads();
        const uint64_t tag = (static_cast<uint64_t>(p.generation) << 32) |
                             static_cast<uint32_t>(kk + 1);
        if (tid == 0) {
            TopkHeader* h = reinterpret_cast<TopkHeader*>(my_rec);
            h->m = mc;
            h->s = s_cta;
            h->count = nlocal;
            __threadfence();
            asm volatile("st.release.gpu.global.b64 [%0], %1;" ::"l"(&h->tag), "l"(tag) : "memory");
        }

        // ---- merge across the team ---------------------------------------------
        if (warp == 0) {
            bool ok = true;
            float m = -INFINITY, s_m = 0.0f;
            if (lane < p.team) {
                const unsigned char* rec =
                    p.xchg + (static_cast<size_t>(team_id * p.team + lane) * kRing + slot) * p.rec_bytes;
                const TopkHeader* h = reinterpret_cast<const TopkHeader*>(rec);
                uint64_t got;
                asm volatile("ld.acquire.gpu.global.b64 %0, [%1];" : "=l"(got) : "l"(&h->tag) : "memory");
                if (got != tag) {
                    const uint64_t t0 = global_timer_ns();
                    for (uint32_t it = 0;; ++it) {
                        __nanosleep(64);
                        asm volatile("ld.acquire.gpu.global.b64 %0, [%1];"
                                     : "=l"(got)
                                     : "l"(&h->tag)
                                     : "memory");
                        if (got == tag) break;
                        if ((it & 15u) == 15u && global_timer_ns() - t0 > kWaitLimitNs) {
                            ok = false;
                            break;
                        }
                    }
                }
                if (ok) {
                    m = __ldcg(&h->m);
                    s_m = __ldcg(&h->s);
                }
            }
            ok = __all_sync(0xffffffffu, ok);
            const float big_m = warp_max(m);
            float s_l = 0.0f;
            if (m != -INFINITY) s_l = ex2_approx((m - big_m) * kLog2e) * s_m;
            const float s_tot = warp_sum_f(s_l);
            if (lane == 0) {
                sc.status = ok ? 0 : 1;
                sc.row_max = big_m;
                sc.row_logs = logf(s_tot);
            }
        }
        __syncthreads();
        if (sc.status != 0) {
            aborted = true;
            break;
        }
        const float big_m = sc.row_max;
        const float logs = sc.row_logs;
        if (p.out_m && member == 0 && tid == 0) {
            p.out_m[row] = big_m;
            p.out_logs[row] = logs;
        }

        // Rank my keys (thread t holds my_keys[t] and my_keys[t + 512])
        // against all G*K published keys, staged through shared memory in
        // tiles; global rank r < K goes to output position r.
        const int total = p.team * K;
        int64_t mine[2] = {kNoKey, kNoKey};
        int grank[2] = {0, 0};
#pragma unroll
        for (int h = 0; h < 2; ++h)
            if (tid + h * kThreads < K) mine[h] = __ldcg(&my_keys[tid + h * kThreads]);
        for (int base = 0; base < total; base += kCandCap) {
            const int n = min(kCandCap, total - base);
            __syncthreads();
            for (int e = tid; e < n; e += kThreads) {
                const int g = (base + e) / K;
                const int r = (base + e) - g * K;
                const unsigned char* rec =
                    p.xchg + (static_cast<size_t>(team_id * p.team + g) * kRing + slot) * p.rec_bytes;
                cand[e] = __ldcg(reinterpret_cast<const int64_t*>(rec + sizeof(TopkHeader)) + r);
            }
            __syncthreads();
#pragma unroll
            for (int h = 0; h < 2; ++h)
                if (mine[h] != kNoKey)
                    for (int e = 0; e < n; ++e) grank[h] += cand[e] > mine[h];
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t key = mine[h];
            if (key != kNoKey && grank[h] < K) {
                const float sv = value_of_key32(static_cast<int32_t>(key >> 32));
                const int col = 0x7FFFFFFF - static_cast<int32_t>(key & 0xFFFFFFFF);
                const float lp = big_m == -INFINITY ? NAN : (sv - big_m) - logs;
                p.out_ids[row * K + grank[h]] = col;
                p.out_lp[row * K + grank[h]] = lp;
            }
        }
        __syncthreads();
    }

    if (aborted && tid == 0) raise_device_error(p.err, 2);
    if (use_tma && tid == 0) {
        for (int64_t seq = consumed; seq < issued; ++seq) {
            const int st = static_cast<int>(seq % p.nstage);
            mbar_wait_bounded(&sc.full[st], static_cast<uint32_t>((seq / p.nstage) & 1));
        }
    }
}


// ---------------------------------------------------------------------------
// Rows longer than a team can stage (more than kMaxTeam chunks of 16384
// columns): one CTA per row, reading the row from global memory in five
// passes. Rows needing this are those the row-statistics passes could not
// finish, or every kept row when k > 64; the passes are
//   1. the row max m, and the histogram of the top 8 bits of the value keys;
//   2. S = sum e^(s - m), and the next 8 bits among the keys that share the
//      chosen top bits; 3-4. the last two bytes the same way (a radix select
//      of the k-th largest value key);
//   5. the keys above that value, and the lowest columns holding it until k
//      keys are collected, in column order.
// The k keys are then ranked by counting and written with the logprob
// s - m - log S.

constexpr int kWideCtasPerSm = 2;

struct WideShared {
    unsigned int hist[256];
    float red[kWarps];
    int ired[kWarps];
    int ncand;
    int bin;
    int need;
    int taken;
    float m;
    float logs;
    int64_t cand[kMaxK];
};

// The row's columns c = base + 4 * tid + q of the chunk at `base` (4 *
// kThreads columns): scaled exactly, -0.0 as +0.0; -inf past the end.
__device__ __forceinline__ void wide_load(const float* xr, int vocab, int base, bool vec,
                                          const ScaledQuotient& sq, float (&s)[4]) {
    const int c0 = base + 4 * threadIdx.x;
    if (vec && c0 + 4 <= vocab) {
        const float4 x = __ldcs(reinterpret_cast<const float4*>(xr + c0));
        s[0] = x.x;
        s[1] = x.y;
        s[2] = x.z;
        s[3] = x.w;
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) s[q] = c0 + q < vocab ? __ldcs(xr + c0 + q) : -INFINITY;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) s[q] = sq.exact(s[q]) + 0.0f;
}

__device__ __forceinline__ uint32_t ukey_of(float s) {
    return static_cast<uint32_t>(key32_of(s)) ^ 0x80000000u;
}

// Add the lane's bin (256: none) to the shared histogram, one atomic per
// distinct bin of the warp.
__device__ __forceinline__ void hist_add(unsigned int* hist, unsigned int bin) {
    const unsigned int peers = __match_any_sync(0xffffffffu, bin);
    if (bin < 256u && (threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
}

__global__ void __launch_bounds__(kThreads, kWideCtasPerSm)
    topk_wide_kernel(const __grid_constant__ TopkParams p) {
    __shared__ WideShared sh;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int K = p.k;
    const int V = p.vocab;
    const bool vec = p.vec != 0;
    const int64_t nlisted = p.row_list ? static_cast<int64_t>(p.row_list[0]) : p.rows;
    for (int64_t j = blockIdx.x; j < nlisted; j += gridDim.x) {
        const int64_t row = p.row_list ? static_cast<int64_t>(p.row_list[64 + j]) : j;
        const int64_t slot = (p.row0 + row) / p.canvas_len;
        if (!p.row_list && p.keep[slot] == 0) continue;
        const float* xr = p.logits + (p.map_row ? static_cast<int64_t>(p.map_row[row]) : row) * p.row_stride;
        const float temp = p.map_temp ? p.map_temp[row] : p.temps[slot];
        const ScaledQuotient sq = ScaledQuotient::of(fmaxf(temp, kTempFloor));

        // ---- radix select of the k-th largest value key, with m and S ----
        uint32_t prefix = 0, pmask = 0;
        int need = K;
        float m = -INFINITY;
        for (int d = 3; d >= 0; --d) {
            for (int b = tid; b < 256; b += kThreads) sh.hist[b] = 0;
            __syncthreads();
            const int shift = 8 * d;
            float acc = d == 3 ? -INFINITY : 0.0f;
            for (int base = 0; base < V; base += 4 * kThreads) {
                float s[4];
                wide_load(xr, V, base, vec, sq, s);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const bool in = base + 4 * tid + q < V;
                    if (d == 3) acc = fmaxf(acc, s[q]);
                    else if (d == 2 && in && m != -INFINITY) acc += ex2_approx((s[q] - m) * kLog2e);
                    const uint32_t u = ukey_of(s[q]);
                    hist_add(sh.hist, in && (u & pmask) == prefix ? (u >> shift) & 0xFFu : 256u);
                }
            }
            if (d == 3) {
                const float wm = warp_max(acc);
                if (lane == 0) sh.red[warp] = wm;
            } else if (d == 2) {
                const float ws = warp_sum_f(acc);
                if (lane == 0) sh.red[warp] = ws;
            }
            __syncthreads();
            if (tid == 0) {
                // the bin holding the need-th largest key under the prefix
                int above = 0, b = 255;
                for (; b > 0; --b) {
                    if (above + static_cast<int>(sh.hist[b]) >= need) break;
                    above += static_cast<int>(sh.hist[b]);
                }
                sh.bin = b;
                sh.need = need - above;
                if (d == 3) {
                    float r = -INFINITY;
                    for (int w = 0; w < kWarps; ++w) r = fmaxf(r, sh.red[w]);
                    sh.m = r;
                } else if (d == 2) {
                    float r = 0.0f;
                    for (int w = 0; w < kWarps; ++w) r += sh.red[w];
                    sh.logs = logf(r);
                }
            }
            __syncthreads();
            prefix |= static_cast<uint32_t>(sh.bin) << shift;
            pmask |= 0xFFu << shift;
            need = sh.need;
            if (d == 3) m = sh.m;
            __syncthreads();
        }
        const uint32_t vt = prefix;  // the k-th largest value key; `need` of its holders are taken

        // ---- the keys: all above vt, the lowest `need` columns holding vt ----
        if (tid == 0) {
            sh.ncand = 0;
            sh.taken = 0;
        }
        __syncthreads();
        for (int base = 0; base < V; base += 4 * kThreads) {
            float s[4];
            wide_load(xr, V, base, vec, sq, s);
            int neq = 0;
            bool eq[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int c = base + 4 * tid + q;
                const uint32_t u = ukey_of(s[q]);
                eq[q] = c < V && u == vt;
                neq += eq[q];
                if (c < V && u > vt) {
                    const int pos = atomicAdd(&sh.ncand, 1);  // < K: fewer than K keys exceed vt
                    if (pos < kMaxK) sh.cand[pos] = make_key(s[q], c);
                }
            }
            // the holders of vt in column order: the warp's, then the CTA's
            int incl = neq;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            if (lane == 31) sh.ired[warp] = incl;
            __syncthreads();
            int before = sh.taken;
            int chunk_total = 0;
            for (int w = 0; w < kWarps; ++w) {
                const int c = sh.ired[w];
                if (w < warp) before += c;
                chunk_total += c;
            }
            int order = before + incl - neq;
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (eq[q]) {
                    if (order < need) {
                        const int pos = atomicAdd(&sh.ncand, 1);
                        if (pos < kMaxK) sh.cand[pos] = make_key(s[q], base + 4 * tid + q);
                    }
                    ++order;
                }
            __syncthreads();
            if (tid == 0) sh.taken += chunk_total;
            __syncthreads();
        }

        // ---- rank the k keys and write them -------------------------------
        const float logs = sh.logs;
        if (p.out_m && tid == 0) {
            p.out_m[row] = m;
            p.out_logs[row] = logs;
        }
        for (int c = tid; c < K; c += kThreads) {
            const int64_t key = sh.cand[c];
            int rank = 0;
            for (int o = 0; o < K; ++o) rank += sh.cand[o] > key;
            const float sv = value_of_key32(static_cast<int32_t>(key >> 32));
            const int col = 0x7FFFFFFF - static_cast<int32_t>(key & 0xFFFFFFFF);
            p.out_ids[row * K + rank] = col;
            p.out_lp[row * K + rank] = m == -INFINITY ? NAN : (sv - m) - logs;
        }
        __syncthreads();
    }
}

namespace {

size_t record_bytes(int k) {
    return (sizeof(TopkHeader) + static_cast<size_t>(k) * 8 + 31) & ~static_cast<size_t>(31);
}

template <int VEC4>
drs_status launch_topk(TopkParams& prm, int grid, size_t smem, cudaStream_t stream) {
    auto kernel = topk_kernel<VEC4>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return DRS_ERR_CUDA;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, smem);
    if (e != cudaSuccess || per_sm < 1) return DRS_ERR_CUDA;
    if (grid > per_sm * sm_count()) return DRS_ERR_UNSUPPORTED;
    void* args[] = {&prm};
    e = cudaLaunchCooperativeKernel(reinterpret_cast<void*>(kernel), dim3(grid), dim3(kThreads),
                                    args, smem, stream);
    return cuda_status(e);
}

}  // namespace

size_t exact_topk_workspace_bytes(int32_t k) {
    if (k <= 0) return 0;
    return static_cast<size_t>(1024) * kRing * record_bytes(k);
}

drs_status exact_topk(const float* logits, int64_t rows, int64_t vocab, int64_t row_stride,
                      int64_t row0, const float* temps, int64_t canvas_len, const uint8_t* keep,
                      const int32_t* row_list, int32_t k, int32_t* out_ids, float* out_logprobs,
                      void* workspace, cudaStream_t stream, const ExactTopkMap* map) {
    const int sms = sm_count();
    if (sms <= 0) return DRS_ERR_CUDA;
    const RowPlan plan = plan_rows(rows, static_cast<int>(vocab), sms, false);
    if (!plan.team) {
        // rows too long for a team: one CTA per row
        TopkParams w{};
        w.logits = logits;
        w.row_stride = row_stride;
        w.rows = rows;
        w.row0 = row0;
        w.row_list = row_list;
        w.temps = temps;
        w.canvas_len = canvas_len;
        w.keep = keep;
        w.out_ids = out_ids;
        w.out_lp = out_logprobs;
        w.k = k;
        w.vocab = static_cast<int32_t>(vocab);
        if (map) {
            w.map_row = map->row;
            w.map_temp = map->temp;
            w.out_m = map->out_m;
            w.out_logs = map->out_logs;
        }
        w.vec = aligned(logits, 16) && (row_stride % 4 == 0) ? 1 : 0;
        const int64_t g = row_list ? static_cast<int64_t>(kWideCtasPerSm) * sms
                                   : std::min<int64_t>(rows, static_cast<int64_t>(kWideCtasPerSm) * sms);
        topk_wide_kernel<<<static_cast<int>(g), kThreads, 0, stream>>>(w);
        return cuda_status(cudaGetLastError());
    }

    TopkParams prm{};
    prm.logits = logits;
    prm.row_stride = row_stride;
    prm.rows = rows;
    prm.row0 = row0;
    prm.row_list = row_list;
    prm.temps = temps;
    prm.canvas_len = canvas_len;
    prm.keep = keep;
    prm.out_ids = out_ids;
    prm.out_lp = out_logprobs;
    prm.xchg = static_cast<unsigned char*>(workspace);
    prm.err = device_error_flag();
    prm.generation = next_generation();
    prm.k = k;
    prm.vocab = static_cast<int32_t>(vocab);
    prm.team = plan.team;
    prm.chunk = plan.chunk;
    prm.num_teams = plan.num_teams;
    prm.rec_bytes = static_cast<int32_t>(record_bytes(k));
    if (map) {
        prm.map_row = map->row;
        prm.map_temp = map->temp;
        prm.out_m = map->out_m;
        prm.out_logs = map->out_logs;
    }
    if (!prm.err) return DRS_ERR_CUDA;

    const bool tma = aligned(logits, 16) && (row_stride % 4 == 0);
    const size_t scratch = ((sizeof(TopkScratch) + 127) & ~static_cast<size_t>(127)) +
                           static_cast<size_t>(kCandCap) * sizeof(int64_t);
    const size_t smem_limit = kSmemPerCta;
    if (tma) {
        prm.stage_bytes = (plan.chunk * 4 + 127) & ~127;
        int ns = static_cast<int>((smem_limit - scratch) / prm.stage_bytes);
        prm.nstage = ns > kMaxStages ? kMaxStages : ns;
        if (prm.nstage < 2) prm.nstage = 0;
    }
    if (!prm.nstage) prm.stage_bytes = 0;
    const size_t smem = static_cast<size_t>(prm.nstage) * prm.stage_bytes + scratch;
    const int grid = plan.team * plan.num_teams;
    return launch_topk<8>(prm, grid, smem, stream);  // plan_rows(..., false): 32 logits per thread
}

int32_t exact_topk_max_k() { return kMaxK; }

}  // namespace drs
