// row_stats.cu -- one-read row statistics of temperature-scaled logits:
// argmax, Gumbel-max sample, softmax entropy and (optionally) the softmax in
// bf16/fp16 (page "vllm.model_executor.models.diffusion_gemma_sampler",
// module docstring, sample_row_stats and sample_row_stats_reference).
//
// Layout of the work. A row of V fp32 logits is split into G contiguous
// chunks of `chunk` columns (a multiple of 4). G CTAs -- a team -- own the G
// chunks of every row of the team; teams take rows round robin. The kernel
// is persistent (one CTA per SM, cooperative launch so that all CTAs are
// resident) and a CTA walks through its team's rows:
//
//   1. A bulk copy (TMA) stages the CTA's chunk of a row in shared memory,
//      several rows ahead; each thread then holds up to 32 logits in
//      registers (float4 slot i of thread t covers columns 4*(i*512+t)+0..3
//      of the chunk, so shared-memory reads and global stores coalesce).
//   2. s = x / max(T, 1e-10) as one IEEE fp32 division per element.
//   3. CTA max m and lowest-column argmax; S = sum e^(s-m) and
//      W = sum e^(s-m)(s-m) (the "online max and sum" of the page).
//   4. Gumbel-max race (T > 0): score = s + g with g from Philox keyed by
//      (seed, row, column). Elements within kNearTop of the max are scored
//      first; their best score B bounds the rest: an element can only win
//      if s > B - 16.64 (the largest possible g), and then only if the
//      exact lower bound 1 - u <= -log u of its exponential variate allows
//      it, so most of the row draws no logarithm.
//   5. The CTA publishes (m, S, W, argmax, best score, best column) in the
//      workspace, waits for the team's G records of the row and merges them
//      (M = max m, S = sum S e^(m-M), W = sum e^(m-M)(W + (m-M) S),
//      entropy = log S - W / S).
//   6. Probabilities e^(s - M - log S) are written from registers, rounded
//      to nearest even.
//
// HBM traffic: every logit is read once (by the bulk copy) and every
// probability written once.
#include <cfloat>
#include <climits>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "drs_device.cuh"
#include "drs_internal.h"

namespace drs {

namespace {

constexpr int kMaxStages = 4;
constexpr float kNearTop = 2.0f;  // first-sweep window below the CTA max

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
    int32_t nstage;     // shared-memory stages (0: no bulk copy)
    int32_t stage_bytes;
    int32_t probs_dtype;
    int32_t probs_vec;  // 8-byte probability stores are aligned
};

struct Scratch {
    uint64_t full[kMaxStages];
    float wmax[kWarps];
    double ws[kWarps];
    double ww[kWarps];
    int warg[kWarps];
    float wbest[2][kWarps];
    int wbcol[2][kWarps];
    float row_max;
    float row_log2s;
    int status;
};

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float max4(const float4& v) {
    return fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
}

__device__ __forceinline__ float comp(const float4& v, int q) {
    return q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w;
}

__device__ __forceinline__ void set_comp(float4& v, int q, float x) {
    if (q == 0) v.x = x;
    else if (q == 1) v.y = x;
    else if (q == 2) v.z = x;
    else v.w = x;
}

__device__ __forceinline__ uint16_t prob_code(float p, int dtype) {
    if (dtype == 1) return __bfloat16_as_ushort(__float2bfloat16_rn(p));
    return __half_as_ushort(__float2half_rn(p));
}

}  // namespace

template <int VEC4, bool kTma>
__global__ void __launch_bounds__(kThreads, 1)
    row_stats_kernel(const __grid_constant__ RowStatsParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    Scratch& sc = *reinterpret_cast<Scratch*>(smem + p.nstage * p.stage_bytes);

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int team_id = blockIdx.x / p.team;
    const int member = blockIdx.x - team_id * p.team;
    const int col0 = member * p.chunk;
    const int ncols = min(p.vocab - col0, p.chunk);
    const int nfull4 = ncols >> 2;
    const uint32_t copy_bytes = static_cast<uint32_t>(nfull4) * 16u;
    const int64_t nrows =
        team_id < p.rows ? (p.rows - 1 - team_id) / p.num_teams + 1 : 0;

    if (kTma && tid == 0) {
        for (int s = 0; s < p.nstage; ++s) mbar_init(&sc.full[s], 1);
        fence_barrier_init();
    }
    __syncthreads();

    auto issue_copy = [&](int64_t seq) {
        const int s = static_cast<int>(seq % p.nstage);
        const int64_t row = team_id + seq * p.num_teams;
        float* dst = reinterpret_cast<float*>(smem + s * p.stage_bytes);
        mbar_arrive_expect_tx(&sc.full[s], copy_bytes);
        if (copy_bytes)
            tma_load_1d(dst, p.logits + row * p.row_stride + col0, copy_bytes, &sc.full[s]);
    };

    int64_t issued = 0;
    if (kTma && tid == 0) {
        for (; issued < nrows && issued < p.nstage; ++issued) issue_copy(issued);
    }

    bool aborted = false;
    int64_t consumed = 0;  // rows whose staged chunk has been read
    for (int64_t k = 0; k < nrows; ++k) {
        const int64_t row = team_id + k * p.num_teams;
        const float* grow = p.logits + row * p.row_stride + col0;

        // ---- 1. load the chunk into registers -----------------------------
        bool timed_out = false;
        const int s = kTma ? static_cast<int>(k % p.nstage) : 0;
        if (kTma) timed_out = !mbar_wait_bounded(&sc.full[s], static_cast<uint32_t>((k / p.nstage) & 1));
        float4 v[VEC4];
        const float4* stage4 = reinterpret_cast<const float4*>(smem + s * p.stage_bytes);
#pragma unroll
        for (int i = 0; i < VEC4; ++i) {
            const int f = i * kThreads + tid;
            float4 x = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            if (f < nfull4) {
                if (kTma) {
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
        consumed = k + 1;
        if (kTma && tid == 0 && issued < nrows) {
            fence_proxy_async_smem();
            issue_copy(issued);
            ++issued;
        }

        // ---- 2. temperature ----------------------------------------------
        const int64_t grow_id = p.row0 + row;  // global row
        const float temp = p.temps[grow_id / p.canvas_len];
        const float te = fmaxf(temp, kTempFloor);
        const bool noisy = temp > 0.0f;
        if (te != 1.0f) {
#pragma unroll
            for (int i = 0; i < VEC4; ++i) {
                v[i].x = __fdiv_rn(v[i].x, te);
                v[i].y = __fdiv_rn(v[i].y, te);
                v[i].z = __fdiv_rn(v[i].z, te);
                v[i].w = __fdiv_rn(v[i].w, te);
            }
        }

        // ---- 3. max, argmax, sums ----------------------------------------
        float mt = -INFINITY;
#pragma unroll
        for (int i = 0; i < VEC4; ++i) mt = fmaxf(mt, max4(v[i]));
        {
            const float wm = warp_max(mt);
            if (lane == 0) sc.wmax[warp] = wm;
        }
        __syncthreads();
        const float mc = warp_max(lane < kWarps ? sc.wmax[lane] : -INFINITY);

        int arg_t = INT_MAX;
        if (mt == mc && mc != -INFINITY) {
#pragma unroll
            for (int i = 0; i < VEC4; ++i) {
                const int f = i * kThreads + tid;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (comp(v[i], q) == mc && arg_t == INT_MAX) arg_t = col0 + 4 * f + q;
            }
        }

        float st = 0.0f, wt = 0.0f;
#pragma unroll
        for (int i = 0; i < VEC4; ++i) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float d = fmaxf(comp(v[i], q) - mc, -1e30f);
                const float e = ex2_approx(d * kLog2e);
                st += e;
                wt = fmaf(e, d, wt);
            }
        }

        // ---- 4a. Gumbel race near the top ----------------------------------
        const bool race = noisy && mc != -INFINITY;
        const float near = mc - kNearTop;
        float bs = -INFINITY;
        int bc = INT_MAX;
        if (race) {
#pragma unroll
            for (int i = 0; i < VEC4; ++i) {
                if (max4(v[i]) >= near) {
                    const int f = i * kThreads + tid;
                    const uint4 w = noise_words(p.key, static_cast<uint64_t>(grow_id),
                                                static_cast<uint64_t>((col0 >> 2) + f));
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float x = comp(v[i], q);
                        if (x >= near) {
                            const float score = x + gumbel_of_bits(word_of(w, q));
                            const int c = col0 + 4 * f + q;
                            if (beats(score, c, bs, bc)) {
                                bs = score;
                                bc = c;
                            }
                        }
                    }
                }
            }
        }

        // CTA reduction of S, W, argmax and the first-sweep best.
        {
            const double ws = warp_sum_d(static_cast<double>(st));
            const double ww = warp_sum_d(static_cast<double>(wt));
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
        const double s_cta = warp_sum_d(lane < kWarps ? sc.ws[lane] : 0.0);
        const double w_cta = warp_sum_d(lane < kWarps ? sc.ww[lane] : 0.0);
        const int arg_cta =
            mc == -INFINITY ? col0 : warp_min_i(lane < kWarps ? sc.warg[lane] : INT_MAX);
        float best = lane < kWarps ? sc.wbest[0][lane] : -INFINITY;
        int best_col = lane < kWarps ? sc.wbcol[0][lane] : INT_MAX;
        warp_best(best, best_col);

        // ---- 4b. Gumbel race over the rest, pruned -------------------------
        if (race) {
            bs = best;
            bc = best_col;
            const float floor_score = best - kGumbelMax;
#pragma unroll
            for (int i = 0; i < VEC4; ++i) {
                const float gm = max4(v[i]);
                if (gm > floor_score) {
                    const int f = i * kThreads + tid;
                    bool any = false;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float x = comp(v[i], q);
                        any |= (x > floor_score && x < near);
                    }
                    if (any) {
                        const uint4 w = noise_words(p.key, static_cast<uint64_t>(grow_id),
                                                    static_cast<uint64_t>((col0 >> 2) + f));
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float x = comp(v[i], q);
                            if (x > floor_score && x < near) {
                                const uint32_t word = word_of(w, q);
                                // x + g >= bs needs -log u <= exp(x - bs); since
                                // 1 - u <= -log u, a larger 1 - u rules it out.
                                const float lim = ex2_approx((x - bs) * kLog2e) * 1.0001f;
                                if (exponential_lower_bound(word) > lim) continue;
                                const float score = x + gumbel_of_bits(word);
                                const int c = col0 + 4 * f + q;
                                if (beats(score, c, bs, bc)) {
                                    bs = score;
                                    bc = c;
                                }
                            }
                        }
                    }
                }
            }
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

        // ---- 5. exchange with the team and merge ----------------------------
        const int slot = static_cast<int>(k % kRing);
        const uint64_t tag = (static_cast<uint64_t>(p.generation) << 32) |
                             static_cast<uint32_t>(k + 1);
        if (tid == 0) {
            publish_partial(p.xchg + static_cast<size_t>(blockIdx.x) * kRing + slot, mc,
                            static_cast<float>(s_cta), static_cast<float>(w_cta), arg_cta,
                            best, best_col, tag);
        }
        if (warp == 0) {
            bool ok = true;
            float m = -INFINITY, s_m = 0.0f, w_m = 0.0f, b_m = -INFINITY;
            int a_m = INT_MAX, bc_m = INT_MAX;
            if (lane < p.team) {
                Partial rp;
                ok = read_partial_bounded(
                    p.xchg + static_cast<size_t>(team_id * p.team + lane) * kRing + slot, tag,
                    rp);
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
            double s_d = 0.0, w_d = 0.0;
            if (m != -INFINITY) {
                const double dm = static_cast<double>(m) - static_cast<double>(big_m);
                const double f = exp(dm);
                s_d = f * static_cast<double>(s_m);
                w_d = f * (static_cast<double>(w_m) + dm * static_cast<double>(s_m));
            }
            const double s_tot = warp_sum_d(s_d);
            const double w_tot = warp_sum_d(w_d);
            const int arg_row = warp_min_i(m == big_m ? a_m : INT_MAX);
            warp_best(b_m, bc_m);
            if (lane == 0) {
                sc.row_max = big_m;
                sc.row_log2s = s_tot > 0.0 ? static_cast<float>(log2(s_tot)) : 0.0f;
                sc.status = ok ? 0 : 1;
                if (ok && member == 0) {
                    const bool drawn = noisy && b_m != -INFINITY;
                    p.argmax[row] = arg_row;
                    p.sample[row] = drawn ? bc_m : arg_row;
                    p.entropy[row] =
                        s_tot > 0.0 ? static_cast<float>(log(s_tot) - w_tot / s_tot) : 0.0f;
                }
            }
        }
        __syncthreads();
        if (sc.status != 0) {
            aborted = true;
            break;
        }

        // ---- 6. probabilities ----------------------------------------------
        if (p.probs_dtype != 0) {
            const float big_m = sc.row_max;
            const float l2s = sc.row_log2s;
            uint16_t* prow = static_cast<uint16_t*>(p.probs) + row * p.probs_row_stride + col0;
#pragma unroll
            for (int i = 0; i < VEC4; ++i) {
                const int f = i * kThreads + tid;
                if (4 * f >= ncols) continue;
                uint16_t code[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float pr;
                    if (big_m == -INFINITY) {
                        pr = NAN;
                    } else {
                        pr = ex2_approx(fmaf(comp(v[i], q) - big_m, kLog2e, -l2s));
                    }
                    code[q] = prob_code(pr, p.probs_dtype);
                }
                if (p.probs_vec && f < nfull4) {
                    const uint2 packed = make_uint2(
                        static_cast<uint32_t>(code[0]) | (static_cast<uint32_t>(code[1]) << 16),
                        static_cast<uint32_t>(code[2]) | (static_cast<uint32_t>(code[3]) << 16));
                    __stcs(reinterpret_cast<uint2*>(prow + 4 * f), packed);
                } else {
                    for (int q = 0; q < 4; ++q)
                        if (4 * f + q < ncols) prow[4 * f + q] = code[q];
                }
            }
        }
    }

    if (aborted && tid == 0) raise_device_error(p.err, 1);
    // Bulk copies still in flight must land before the CTA's shared memory
    // is released.
    if (kTma && tid == 0) {
        for (int64_t seq = consumed; seq < issued; ++seq) {
            const int st = static_cast<int>(seq % p.nstage);
            mbar_wait_bounded(&sc.full[st], static_cast<uint32_t>((seq / p.nstage) & 1));
        }
    }
}

namespace {

template <int VEC4, bool kTma>
drs_status launch_row_stats(RowStatsParams& prm, int grid, size_t smem,
                            cudaStream_t stream) {
    auto kernel = row_stats_kernel<VEC4, kTma>;
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

extern "C" size_t drs_row_stats_workspace_bytes(int64_t rows, int64_t vocab) {
    (void)rows;
    (void)vocab;
    // One ring of exchange records per resident CTA, for up to 1024 CTAs.
    return static_cast<size_t>(1024) * drs::kRing * sizeof(drs::Partial);
}

extern "C" drs_status drs_row_stats(const float* logits, int64_t rows, int64_t vocab,
                                    int64_t row_stride, const float* temps,
                                    int64_t canvas_len, uint64_t seed, int64_t row0,
                                    int64_t* argmax,
                                    int64_t* sample, float* entropy,
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
    const int capacity = sms < 1024 ? sms : 1024;
    const RowPlan plan = plan_rows(rows, static_cast<int>(vocab), capacity);
    if (!plan.team) return DRS_ERR_UNSUPPORTED;

    const bool tma = aligned(logits, 16) && (row_stride % 4 == 0);
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
    if (!prm.err) return DRS_ERR_CUDA;

    const size_t scratch = (sizeof(Scratch) + 127) & ~static_cast<size_t>(127);
    const size_t smem_limit = 227 * 1024;
    if (tma) {
        prm.stage_bytes = (plan.chunk * 4 + 127) & ~127;
        int ns = static_cast<int>((smem_limit - scratch) / prm.stage_bytes);
        if (ns > kMaxStages) ns = kMaxStages;
        prm.nstage = ns;
    }
    const bool use_tma = tma && prm.nstage >= 2;
    if (!use_tma) {
        prm.nstage = 0;
        prm.stage_bytes = 0;
    }
    const size_t smem = static_cast<size_t>(prm.nstage) * prm.stage_bytes + scratch;
    const int grid = plan.team * plan.num_teams;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (plan.vec4 == 4) {
        return use_tma ? launch_row_stats<4, true>(prm, grid, smem, st)
                       : launch_row_stats<4, false>(prm, grid, smem, st);
    }
    return use_tma ? launch_row_stats<8, true>(prm, grid, smem, st)
                   : launch_row_stats<8, false>(prm, grid, smem, st);
}
