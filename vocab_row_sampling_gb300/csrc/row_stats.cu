// row_stats.cu -- one-read row statistics of temperature-scaled logits:
// argmax, Gumbel-max sample, softmax entropy and (optionally) the softmax in
// bf16/fp16 (page "vllm.model_executor.models.diffusion_gemma_sampler",
// module docstring, sample_row_stats and sample_row_stats_reference).
//
// Layout of the work. A row of V fp32 logits is split into G contiguous
// chunks of `chunk` columns (a multiple of 4). G CTAs -- a team -- own the G
// chunks of every row of the team; teams take rows round robin. The kernel
// is persistent (cooperative launch, so all CTAs are resident; two CTAs per
// SM in the 16-logit layout so that one computes while the other waits) and
// a CTA walks through its team's rows:
//
//   1. A bulk copy (TMA) stages the CTA's chunk of a row in shared memory,
//      several rows ahead; each thread then holds its logits in registers
//      (float4 slot i of thread t covers columns 4*(i*512+t)+0..3 of the
//      chunk, so shared-memory reads and global stores coalesce).
//   2. s = x / max(T, 1e-10): the IEEE fp32 quotient, from a per-row
//      reciprocal and two FMA corrections (ScaledQuotient).
//   3. CTA max m and lowest-column argmax; S = sum e^(s-m) and
//      W = sum e^(s-m)(s-m) (the "online max and sum" of the page).
//   4. Gumbel-max race (T > 0), score = s + g with g from Philox keyed by
//      (seed, row, column). Elements within kNearTop of the max are scored
//      exactly first; their best B bounds the rest: an element can only win
//      if s > B - 16.64 (the largest possible g), and then only if the exact
//      bound 1 - u <= -log u of its exponential variate allows it. Only the
//      few survivors take logarithms, in one rolled loop.
//   5. The CTA publishes (m, S, W, argmax, best score, best column) in the
//      workspace, waits for the team's G records of the row and merges them
//      (M = max m, S = sum S e^(m-M), W = sum e^(m-M)(W + (m-M) S),
//      entropy = log S - W / S).
//   6. Probabilities e^(s - M - log S) are written from registers, rounded
//      to nearest even.
//
// HBM traffic: every logit is read once (by the bulk copy) and every
// probability written once. No fp64 arithmetic (its rate on GB300 is a
// small fraction of fp32's).
#include <cfloat>
#include <climits>
#include <atomic>
#include <mutex>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "drs_device.cuh"
#include "drs_internal.h"

namespace drs {

namespace {

constexpr int kMaxStages = 3;
constexpr float kNearTop = 2.0f;  // window below the CTA max scored exactly first

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
    Partial* xchg;
    int* err;
    PhiloxKey key;
    uint32_t generation;
    int32_t vocab;
    int32_t team;       // CTAs per row
    int32_t chunk;      // columns per CTA (multiple of 4)
    int32_t num_teams;
    int32_t nstage;     // shared-memory stages, one chunk each (>= 3)
    int32_t stage_bytes;
    int32_t use_tma;    // stages filled by bulk copies (rows 16-byte aligned)
    int32_t probs_dtype;
    int32_t probs_vec;  // 8-byte probability stores are aligned
    int32_t fault;      // test hook: CTA 0 withholds its first record
};

// Test hook state: the next launch withholds one record (see
// drs_test_inject_fault).
std::atomic<int> g_inject_fault{0};

struct Scratch {
    uint64_t full[kMaxStages];
    float wmax[kWarps];
    int wflag[kWarps];
    float ws[kWarps];
    float ww[kWarps];
    int warg[kWarps];
    float wbest[2][kWarps];
    int wbcol[2][kWarps];
    float row_max;
    float row_log2s;
    int status;
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

// log2(1.0001): the race's bound e^(s - best) is widened by 1e-4 so that
// rounding in it never prunes an element whose fp32 score could win.
constexpr float kRaceMarginLog2 = 1.4426229e-4f;

}  // namespace

template <int VEC4>
__global__ void __launch_bounds__(kThreads, VEC4 == 4 ? 2 : 1)
    row_stats_kernel(const __grid_constant__ RowStatsParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    Scratch& sc = *reinterpret_cast<Scratch*>(smem + p.nstage * p.stage_bytes);
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
    const int64_t nrows = team_id < p.rows ? (p.rows - 1 - team_id) / p.num_teams + 1 : 0;
    // Stage of row k: k % nstage. Without bulk copies the scaled logits of
    // a row still wait in "stage" buffers for the next iteration's
    // finalisation, so nstage >= 2 in both modes.
    const int nstage = p.nstage;

    if (use_tma && tid == 0) {
        for (int s = 0; s < nstage; ++s) mbar_init(&sc.full[s], 1);
        fence_barrier_init();
    }
    __syncthreads();

    int64_t issued = 0;  // rows whose chunk copy was issued (thread 0 only)
    auto issue_copy = [&]() {
        const int s = static_cast<int>(issued % nstage);
        const int64_t row = team_id + issued * p.num_teams;
        mbar_arrive_expect_tx(&sc.full[s], copy_bytes);
        if (copy_bytes)
            tma_load_1d(smem + s * p.stage_bytes, p.logits + row * p.row_stride + col0, copy_bytes,
                        &sc.full[s]);
        ++issued;
    };
    if (use_tma && tid == 0) {
        while (issued < nrows && issued < nstage) issue_copy();
    }

    bool aborted = false;
    int64_t consumed = 0;
    bool prev_noisy = false;
    // Iteration k computes row k's partials (A) and then finalises row k-1
    // (F): the team's records of row k-1 were published one row of work ago,
    // so the exchange latency hides behind A(k).
    for (int64_t k = 0; k <= nrows; ++k) {
        bool cur_noisy = false;
        if (k < nrows) {
            const int64_t row = team_id + k * p.num_teams;
            const int64_t grow_id = p.row0 + row;  // global row
            const float* grow = p.logits + row * p.row_stride + col0;
            const int s = static_cast<int>(k % nstage);
            float4* stage4 = reinterpret_cast<float4*>(smem + s * p.stage_bytes);

            // ---- A1. load the chunk into registers ---------------------------
            bool timed_out = false;
            if (use_tma)
                timed_out = !mbar_wait_bounded(&sc.full[s], static_cast<uint32_t>((k / nstage) & 1));
            float4 v[VEC4];
#pragma unroll
            for (int i = 0; i < VEC4; ++i) {
                const int f = i * kThreads + tid;
                float4 x = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
                if (i * kThreads < nslot4) {  // CTA-uniform: slot i holds columns somewhere
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

            // ---- A2. temperature ----------------------------------------------
            const float temp = p.temps[grow_id / p.canvas_len];  // CTA-uniform
            const ScaledQuotient sq = ScaledQuotient::of(fmaxf(temp, kTempFloor));
            const bool noisy = temp > 0.0f;
            cur_noisy = noisy;
            sq.apply(v, nslot4);

            // ---- A3. CTA max ---------------------------------------------------
            float mt = -INFINITY;
#pragma unroll
            for (int i = 0; i < VEC4; ++i) mt = fmaxf(mt, max4(v[i]));
            {
                const float wm = warp_max(mt);
                const int wf = __any_sync(0xffffffffu, timed_out);
                if (lane == 0) {
                    sc.wmax[warp] = wm;
                    sc.wflag[warp] = wf;
                }
            }
            __syncthreads();
            if (__any_sync(0xffffffffu, lane < kWarps && sc.wflag[lane])) {
                aborted = true;
                break;
            }
            consumed = k + 1;
            // The stage of row k-2 was read for the last time in iteration
            // k-1: it now takes row k+1.
            if (use_tma && tid == 0 && k >= 2 && issued < nrows) {
                fence_proxy_async_smem();
                issue_copy();
            }
            float mc = warp_max(lane < kWarps ? sc.wmax[lane] : -INFINITY);

            // Exactness guard: the corrected quotient is exact inside
            // ScaledQuotient::fast_ok. A CTA max outside it (zero, subnormal,
            // huge, or a tiny dividend) decides the argmax among values that
            // may round differently, so the chunk is re-read from global
            // memory and divided exactly (CTA-uniform, rare).
            if (sq.mode == ScaledQuotient::kDivide && mc != -INFINITY &&
                !ScaledQuotient::fast_ok(mc * sq.t, mc)) {
                mt = -INFINITY;
#pragma unroll
                for (int i = 0; i < VEC4; ++i) {
                    const int f = i * kThreads + tid;
                    if (i * kThreads < nslot4 && f < nslot4) {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            if (4 * f + q < ncols) set_comp(v[i], q, sq.exact(grow[4 * f + q]));
                    }
                    mt = fmaxf(mt, max4(v[i]));
                }
                __syncthreads();
                {
                    const float wm = warp_max(mt);
                    if (lane == 0) sc.wmax[warp] = wm;
                }
                __syncthreads();
                mc = warp_max(lane < kWarps ? sc.wmax[lane] : -INFINITY);
            }
            // The scaled logits wait in the stage for the finalisation of the
            // row in the next iteration (each thread rewrites its own slots).
#pragma unroll
            for (int i = 0; i < VEC4; ++i) {
                const int f = i * kThreads + tid;
                if (i * kThreads < nslot4 && f < nslot4) stage4[f] = v[i];
            }

            // ---- A4. argmax, sums, exact race near the top --------------------
            // Only threads holding a value within kNearTop of the CTA max look
            // for the argmax and the near-top elements.
            const bool race = noisy && mc != -INFINITY;
            const float near = mc - kNearTop;
            int arg_t = INT_MAX;
            uint32_t near_mask = 0;
            if (mt >= near && mc != -INFINITY) {
#pragma unroll
                for (int i = 0; i < VEC4; ++i)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float x = comp(v[i], q);
                        if (x == mc && arg_t == INT_MAX) arg_t = col0 + 4 * (i * kThreads + tid) + q;
                        if (x >= near) near_mask |= 1u << (4 * i + q);
                    }
            }
            float st = 0.0f, wt = 0.0f;
#pragma unroll
            for (int i = 0; i < VEC4; ++i) {
                if (i * kThreads < nslot4) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float d = fmaxf(comp(v[i], q) - mc, -1e30f);  // -inf, NaN -> e = 0
                        const float e = ex2_approx(d * kLog2e);
                        st += e;
                        wt = fmaf(e, d, wt);
                    }
                }
            }
            float bs = -INFINITY;
            int bc = INT_MAX;
            if (race && near_mask) race_exact(v, near_mask, col0, tid, grow_id, p.key, bs, bc);
            {
                const float ws = warp_sum_f(st);
                const float ww = warp_sum_f(wt);
                const int wa = warp_min_i(arg_t);
                float wbs = bs;
                int wbc = bc;
                warp_best(wbs, wbc);
                if (lane == 0) {
                    sc.ws[warp] = ws;
                    sc.ww[warp] = ww;
                    sc.warg[warp] = wa;
                    sc.wbest[0][warp] = wbs;
                    sc.wbcol[0][warp] = wbc;
                }
            }
            __syncthreads();
            const float s_cta = warp_sum_f(lane < kWarps ? sc.ws[lane] : 0.0f);
            const float w_cta = warp_sum_f(lane < kWarps ? sc.ww[lane] : 0.0f);
            const int arg_cta =
                mc == -INFINITY ? col0 : warp_min_i(lane < kWarps ? sc.warg[lane] : INT_MAX);
            float best = lane < kWarps ? sc.wbest[0][lane] : -INFINITY;
            int best_col = lane < kWarps ? sc.wbcol[0][lane] : INT_MAX;
            warp_best(best, best_col);

            // ---- A5. pruned race over the rest ----------------------------------
            // An element can beat `best` only if s > best - 16.64, and then
            // only if 1 - u (a lower bound of -log u) is at most e^(s - best).
            // A float4 group is first tested as a whole (its largest s, its
            // largest word); the few groups that pass are tested element by
            // element, and the survivors scored exactly.
            if (race) {
                bs = best;
                bc = best_col;
                const float floor_score = best - kGumbelMax;
                uint32_t survivors = 0;
#pragma unroll
                for (int i = 0; i < VEC4; ++i) {
                    const float gm = max4(v[i]);
                    if (i * kThreads < nslot4 && gm > floor_score) {
                        const int f = i * kThreads + tid;
                        const uint4 w = noise_words(p.key, static_cast<uint64_t>(grow_id),
                                                    static_cast<uint64_t>((col0 >> 2) + f));
                        const uint32_t wmax = max(max(w.x, w.y), max(w.z, w.w));
                        const float lim_g = ex2_approx(fmaf(gm - best, kLog2e, kRaceMarginLog2));
                        if (one_minus_u_lower(wmax) <= lim_g) {
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const float x = comp(v[i], q);
                                const float lim =
                                    ex2_approx(fmaf(x - best, kLog2e, kRaceMarginLog2));
                                if (!((near_mask >> (4 * i + q)) & 1u) && x > floor_score &&
                                    one_minus_u_lower(word_of(w, q)) <= lim)
                                    survivors |= 1u << (4 * i + q);
                            }
                        }
                    }
                }
                if (survivors) race_exact(v, survivors, col0, tid, grow_id, p.key, bs, bc);
                float wbs = bs;
                int wbc = bc;
                warp_best(wbs, wbc);
                if (lane == 0) {
                    sc.wbest[1][warp] = wbs;
                    sc.wbcol[1][warp] = wbc;
                }
                __syncthreads();
                best = lane < kWarps ? sc.wbest[1][lane] : -INFINITY;
                best_col = lane < kWarps ? sc.wbcol[1][lane] : INT_MAX;
                warp_best(best, best_col);
            }

            // ---- A6. publish the CTA's partial of row k -------------------------
            if (tid == 0 && !(p.fault && blockIdx.x == 0 && k == 0)) {
                const uint64_t tag = (static_cast<uint64_t>(p.generation) << 32) |
                                     static_cast<uint32_t>(k + 1);
                publish_partial(p.xchg + static_cast<size_t>(blockIdx.x) * kRing + (k & (kRing - 1)),
                                mc, s_cta, w_cta, arg_cta, best, best_col, tag);
            }
        }

        if (k == 0) {
            prev_noisy = cur_noisy;
            continue;
        }

        // ---- F1. merge the team's records of row k-1 -----------------------------
        const int64_t kf = k - 1;
        const int64_t frow = team_id + kf * p.num_teams;
        if (warp == 0) {
            const uint64_t tag = (static_cast<uint64_t>(p.generation) << 32) |
                                 static_cast<uint32_t>(kf + 1);
            bool ok = true;
            float m = -INFINITY, s_m = 0.0f, w_m = 0.0f, b_m = -INFINITY;
            int a_m = INT_MAX, bc_m = INT_MAX;
            if (lane < p.team) {
                Partial rp;
                ok = read_partial_bounded(p.xchg + static_cast<size_t>(team_id * p.team + lane) * kRing +
                                              (kf & (kRing - 1)),
                                          tag, rp);
                if (ok) {
                    m = rp.m;
                    s_m = rp.s;
                    w_m = rp.w;
                    a_m = rp.arg;
                    b_m = rp.best;
                    bc_m = rp.best_col;
                }
            }
            ok = __all_sync(0xffffffffu, ok);
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
                sc.row_max = big_m;
                sc.row_log2s = s_tot > 0.0f ? log2f(s_tot) : 0.0f;
                sc.status = ok ? 0 : 1;
                if (ok && member == 0) {
                    const bool drawn = prev_noisy && b_m != -INFINITY;
                    p.argmax[frow] = arg_row;
                    p.sample[frow] = drawn ? bc_m : arg_row;
                    p.entropy[frow] = s_tot > 0.0f ? logf(s_tot) - w_tot / s_tot : 0.0f;
                }
            }
        }
        prev_noisy = cur_noisy;
        __syncthreads();
        if (sc.status != 0) {
            aborted = true;
            break;
        }

        // ---- F2. probabilities of row k-1 from its stage -------------------------
        if (p.probs_dtype != 0) {
            const float big_m = sc.row_max;
            const float l2s = sc.row_log2s;
            const bool bf16 = p.probs_dtype == 1;
            const float4* fstage =
                reinterpret_cast<const float4*>(smem + static_cast<int>(kf % nstage) * p.stage_bytes);
            uint16_t* prow = static_cast<uint16_t*>(p.probs) + frow * p.probs_row_stride + col0;
#pragma unroll
            for (int i = 0; i < VEC4; ++i) {
                const int f = i * kThreads + tid;
                if (i * kThreads >= nslot4 || f >= nslot4) continue;
                const float4 sv = fstage[f];
                float pr[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    // e^(s - M - log S) = 2^((s - M) log2 e - log2 S); -inf
                    // columns (and the NaN quotient of -inf) clamp to 0.
                    const float t = fmaxf(fmaf(comp(sv, q) - big_m, kLog2e, -l2s), -256.0f);
                    pr[q] = ex2_approx(t);
                }
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

    if (aborted && tid == 0) raise_device_error(p.err, 1);
    // Bulk copies still in flight must land before the CTA's shared memory
    // is released.
    if (use_tma && tid == 0) {
        for (int64_t seq = consumed; seq < issued; ++seq) {
            const int st = static_cast<int>(seq % nstage);
            mbar_wait_bounded(&sc.full[st], static_cast<uint32_t>((seq / nstage) & 1));
        }
    }
}

namespace {

template <int VEC4>
drs_status launch_row_stats(RowStatsParams& prm, int grid, size_t smem, cudaStream_t stream) {
    auto kernel = row_stats_kernel<VEC4>;
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
    // One ring of exchange records per resident CTA, for up to 1024 CTAs.
    return static_cast<size_t>(1024) * drs::kRing * sizeof(drs::Partial);
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
    const RowPlan plan = plan_rows(rows, static_cast<int>(vocab), sms);
    if (!plan.team) return DRS_ERR_UNSUPPORTED;

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
    prm.xchg = static_cast<Partial*>(workspace);
    prm.err = device_error_flag();
    prm.key = PhiloxKey{static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32)};
    prm.generation = next_generation();
    prm.vocab = static_cast<int32_t>(vocab);
    prm.team = plan.team;
    prm.chunk = plan.chunk;
    prm.num_teams = plan.num_teams;
    prm.probs_dtype = static_cast<int32_t>(probs_dtype);
    prm.probs_vec = probs && aligned(probs, 8) && (probs_row_stride % 4 == 0);
    prm.fault = g_inject_fault.exchange(0);
    if (!prm.err) return DRS_ERR_CUDA;

    // Shared memory: stages of one chunk each (filled by bulk copies when
    // rows start 16-byte aligned; in every case they keep a row's scaled
    // logits until its finalisation) plus the reduction scratch, within the
    // per-CTA share of the SM. Three stages: the row being computed, the row
    // waiting for the team, the row being loaded.
    const bool tma = aligned(logits, 16) && (row_stride % 4 == 0);
    const size_t scratch = (sizeof(Scratch) + 127) & ~static_cast<size_t>(127);
    const size_t smem_limit = smem_per_cta(plan.ctas_per_sm);
    prm.stage_bytes = (plan.chunk * 4 + 127) & ~127;
    int ns = static_cast<int>((smem_limit - scratch) / prm.stage_bytes);
    if (ns > kMaxStages) ns = kMaxStages;
    if (ns < 3) return DRS_ERR_UNSUPPORTED;
    prm.nstage = ns;
    prm.use_tma = tma ? 1 : 0;
    const size_t smem = static_cast<size_t>(prm.nstage) * prm.stage_bytes + scratch;
    const int grid = plan.team * plan.num_teams;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return plan.vec4 == 4 ? launch_row_stats<4>(prm, grid, smem, st)
                          : launch_row_stats<8>(prm, grid, smem, st);
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

constexpr size_t kNoallocWorkspaceBytes = static_cast<size_t>(1024) * drs::kRing * sizeof(drs::Partial);
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
