// stash.cu -- the stash of converged requests' logprobs (page
// "vllm.model_executor.models.diffusion_gemma_sampler": the
// stash_converged_logprobs docstring).
//
// Request j owns logits rows src[j] * canvas_len + p for p < valid[j],
// scaled by clamp(temps[j], 1e-10). Where keep[j], stash row (slots[j], p)
// of the outputs receives `width` columns of (id, value): the argmax, then
// the request's token ids if it has any (num_token_ids[j] > 0), else the
// num_topk largest (value descending, lower id first), then id 0 at -inf.
// The value is the logprob s - max - log(sum e^(s - max)), or the scaled
// logit s in logits mode; out_ranks holds one rank per stash row (below).
//
// Kernels, in stream order:
//   list   one CTA over the (request, position) pairs: the stash rows to
//          write, each with its logits row, temperature, output row and
//          request; for the row kernels also their row list, its header and
//          each entry's RowTemp (their own list kernel is skipped);
//   top-k  k = max(num_topk, 1) keys per entry (the first is the argmax:
//          keys order by value, then by lower column), with each entry's max
//          and log-sum: for k <= 64 the one-read top-k of row_split.cu over
//          the listed rows (pass 1, the merge's threshold, the gather of the
//          warps that reach it; the list as a row map), then the exact
//          kernel on the rows it leaves; for larger k the exact kernel on
//          every entry;
//   write  one warp per entry: the row's columns; in logprobs mode a top-k
//          column's value is the top-k's own logprob (the same arithmetic),
//          any other value one IEEE division.
// Rows of requests that are not kept are never read.
#include <cfloat>
#include <climits>

#include "drs_device.cuh"
#include "drs_internal.h"
#include "row_common.cuh"

namespace drs {
namespace {

constexpr int kListOffset = 64;  // list: count at [0], entries from [64]

struct StashParams {
    const float* logits;
    int64_t row_stride;
    int64_t logits_rows;
    int32_t vocab;
    int64_t canvas_len;
    int64_t requests;
    int64_t out_slots;
    const int32_t* src;
    const int32_t* slots;
    const uint8_t* keep;
    const int32_t* valid;
    const float* temps;
    int32_t num_topk;
    int32_t kq;  // keys per entry from the top-k: max(num_topk, 1)
    const int32_t* num_token_ids;
    const int32_t* token_ids;
    int64_t ids_stride;
    int32_t width;
    int32_t logits_mode;
    int32_t* out_ids;
    float* out_vals;
    int32_t* out_ranks;
    int32_t* list;
    // the row kernels' row list, header and RowTemps (null: the exact kernel
    // takes every entry)
    int32_t* pass_list;
    int32_t* pass_header;
    rs::RowTemp* pass_rt;
    const float* top_lp;
    int32_t* map_row;
    float* map_temp;
    int64_t* map_out;
    int32_t* map_req;
    const int32_t* top_ids;
    const float* row_m;
    const float* row_logs;
};

// The list of kept (request, position) pairs, in order: one CTA walks the
// pairs kListThreads * kListPer at a time, a thread kListPer consecutive
// ones (their loads in flight together), and places its kept pairs after
// the kept pairs before them (a block-wide scan of the counts), so that the
// list, and how the row kernels divide it among themselves, is the same on
// every run.
constexpr int kListThreads = 1024;
constexpr int kListPer = 2;

__global__ void __launch_bounds__(kListThreads) stash_list(const __grid_constant__ StashParams p) {
    __shared__ int wpre[kListThreads / 32];
    __shared__ int wtot;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int n = static_cast<int>(p.requests * p.canvas_len);  // below 2^31 (checked on the host)
    const int cl = static_cast<int>(p.canvas_len);
    int base = 0;
    for (int i0 = 0; i0 < n; i0 += kListThreads * kListPer) {
        bool take[kListPer];
        int req[kListPer];
        float temp[kListPer];
        int64_t row[kListPer], out[kListPer];
        int cnt = 0;
#pragma unroll
        for (int q = 0; q < kListPer; ++q) {
            const int idx = i0 + threadIdx.x * kListPer + q;
            take[q] = false;
            req[q] = 0;
            temp[q] = 0.0f;
            row[q] = out[q] = 0;
            if (idx < n) {
                const int j = idx / cl;
                const int pos = idx - j * cl;
                req[q] = j;
                temp[q] = p.temps[j];
                row[q] = static_cast<int64_t>(p.src[j]) * cl + pos;
                out[q] = static_cast<int64_t>(p.slots[j]) * cl + pos;
                // rows outside the logits or the stash are skipped, never touched
                take[q] = p.keep[j] != 0 && pos < p.valid[j] && p.src[j] >= 0 && row[q] < p.logits_rows &&
                          p.slots[j] >= 0 && p.slots[j] < p.out_slots;
            }
            cnt += take[q] ? 1 : 0;
        }
        // the block's exclusive scan of the counts: within the warp, then
        // over the warps' totals
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) wpre[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int wv = wpre[lane];
            int wi = wv;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, wi, o);
                if (lane >= o) wi += y;
            }
            wpre[lane] = wi - wv;
            if (lane == 31) wtot = wi;
        }
        __syncthreads();
        int e = base + wpre[warp] + (incl - cnt);
#pragma unroll
        for (int q = 0; q < kListPer; ++q) {
            if (!take[q]) continue;
            p.list[kListOffset + e] = e;
            p.map_row[e] = static_cast<int32_t>(row[q]);
            p.map_temp[e] = temp[q];
            p.map_out[e] = out[q];
            p.map_req[e] = req[q];
            if (p.pass_rt) {
                const ScaledQuotient sq = ScaledQuotient::of(fmaxf(temp[q], kTempFloor));
                p.pass_rt[e] = rs::RowTemp{temp[q], sq.t, sq.y, sq.mode};
                p.pass_list[e] = e;
            }
            ++e;
        }
        base += wtot;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        p.list[0] = base;
        if (p.pass_header) {
            p.pass_header[0] = 0;  // the hard-row count
            p.pass_header[rs::kCount1] = base;
        }
    }
}

constexpr int kWriteWarps = 8;

__global__ void __launch_bounds__(kWriteWarps * 32) stash_write(const __grid_constant__ StashParams p) {
    const int lane = threadIdx.x & 31;
    const int64_t e = static_cast<int64_t>(blockIdx.x) * kWriteWarps + (threadIdx.x >> 5);
    if (e >= p.requests * p.canvas_len) return;
    // the entry's fields load beside the list's length (an entry past it
    // holds stale values, never used); the list kernel wrote them, so they
    // load while the exact kernel before this one still runs (a
    // programmatic dependent launch); its results only after it completes
    const int count = p.list[0];
    const int j = p.map_req[e];
    const int64_t out = p.map_out[e];
    const int64_t lrow = p.map_row[e];
    const float te = fmaxf(p.map_temp[e], kTempFloor);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const float big_m = p.row_m[e];
    const float logs = p.row_logs[e];
    const int32_t* keys = p.top_ids + e * p.kq;
    const float* lps = p.top_lp + e * p.kq;
    if (e >= count) return;
    const float* xr = p.logits + lrow * p.row_stride;
    // a request's list holds ids_stride ids at most: a larger count reads no
    // further (the columns past the list are padding)
    const int n_ids = p.token_ids && p.num_token_ids
                          ? static_cast<int>(min(static_cast<int64_t>(p.num_token_ids[j]), p.ids_stride))
                          : 0;
    for (int c = lane; c < p.width; c += 32) {
        int id = 0;
        int kidx = -1;  // the column's place in the top-k, if it has one
        bool has = true;
        if (c == 0) {
            id = keys[0];
            kidx = 0;
        } else if (n_ids > 0) {
            has = c - 1 < n_ids;
            if (has) id = p.token_ids[static_cast<int64_t>(j) * p.ids_stride + (c - 1)];
        } else {
            has = c - 1 < p.num_topk;
            if (has) {
                id = keys[c - 1];
                kidx = c - 1;
            }
        }
        float v;
        if (!has) {
            id = 0;
            v = -INFINITY;
        } else if (id < 0 || id >= p.vocab) {
            v = NAN;  // a token id outside the vocabulary
        } else if (kidx >= 0 && !p.logits_mode) {
            v = lps[kidx];  // (s - max) - log S of the same exact quotient s
        } else {
            const float s = __fdiv_rn(xr[id], te) + 0.0f;
            v = p.logits_mode ? s : (big_m == -INFINITY ? NAN : (s - big_m) - logs);
        }
        p.out_ids[out * p.width + c] = id;
        p.out_vals[out * p.width + c] = v;
    }
    // the rank of column 0's token, 1 + #{columns whose scaled logit exceeds
    // it}: column 0 is the argmax, so none does
    if (lane == 0) p.out_ranks[out] = 1;
}

struct StashLayout {
    size_t list, map_row, map_temp, map_out, map_req, top_ids, top_lp, row_m, row_logs, split, exact,
        total;
};

size_t round_up(size_t n, size_t a) { return (n + a - 1) / a * a; }

StashLayout stash_layout(int64_t requests, int64_t canvas_len, int64_t vocab, int32_t kq) {
    const size_t R = static_cast<size_t>(requests * canvas_len);
    const size_t K = static_cast<size_t>(kq);
    StashLayout l{};
    size_t at = 0;
    auto take = [&](size_t bytes) {
        const size_t here = at;
        at += round_up(bytes, kWorkspaceAlign);
        return here;
    };
    l.list = take(4 * (kListOffset + R));
    l.map_row = take(4 * R);
    l.map_temp = take(4 * R);
    l.map_out = take(8 * R);
    l.map_req = take(4 * R);
    l.top_ids = take(4 * R * K);
    l.top_lp = take(4 * R * K);
    l.row_m = take(4 * R);
    l.row_logs = take(4 * R);
    l.split = take(kq <= split_max_k() ? split_workspace_bytes(static_cast<int64_t>(R), vocab, kq, 1) : 0);
    l.exact = take(exact_topk_workspace_bytes(kq));
    l.total = at;
    return l;
}

}  // namespace
}  // namespace drs

extern "C" size_t drs_stash_workspace_bytes(int64_t requests, int64_t canvas_len, int64_t vocab,
                                            int32_t num_topk) {
    using namespace drs;
    if (requests < 0 || canvas_len < 1 || vocab < 1 || num_topk < 0 ||
        num_topk > exact_topk_max_k())
        return 0;
    if (requests > INT32_MAX / canvas_len) return 0;
    return stash_layout(requests, canvas_len, vocab, num_topk > 0 ? num_topk : 1).total;
}

extern "C" drs_status drs_stash_converged_logprobs(
    const float* logits, int64_t logits_rows, int64_t vocab, int64_t row_stride, int64_t canvas_len,
    int64_t requests, const int32_t* src, const int32_t* slots, const uint8_t* keep,
    const int32_t* valid, const float* temps, int32_t num_topk, const int32_t* num_token_ids,
    const int32_t* token_ids, int64_t ids_stride, int64_t out_slots, int32_t width,
    int32_t* out_ids, float* out_logprobs, int32_t* out_ranks, int logits_mode, void* workspace,
    size_t workspace_bytes, void* stream) {
    using namespace drs;
    if (requests < 0 || logits_rows < 0 || canvas_len < 1 || out_slots < 0)
        return DRS_ERR_INVALID_ARG;
    if (vocab < 1 || row_stride < vocab) return DRS_ERR_INVALID_ARG;
    if (vocab > DRS_MAX_VOCAB) return DRS_ERR_UNSUPPORTED;
    if (num_topk < 0 || num_topk > vocab || num_topk > exact_topk_max_k()) return DRS_ERR_INVALID_ARG;
    if (width < 1 || width < num_topk + 1) return DRS_ERR_INVALID_ARG;
    if (token_ids && (!num_token_ids || ids_stride < 1)) return DRS_ERR_INVALID_ARG;
    if (requests > INT32_MAX / canvas_len || logits_rows > INT32_MAX) return DRS_ERR_UNSUPPORTED;
    if (requests == 0) return DRS_OK;
    if (!logits || !src || !slots || !keep || !valid || !temps || !out_ids || !out_logprobs ||
        !out_ranks)
        return DRS_ERR_INVALID_ARG;
    if (!aligned(logits, 4)) return DRS_ERR_INVALID_ARG;
    const size_t need = drs_stash_workspace_bytes(requests, canvas_len, vocab, num_topk);
    if (!workspace || workspace_bytes < need || !aligned(workspace, kWorkspaceAlign))
        return DRS_ERR_INVALID_ARG;

    const int32_t kq = num_topk > 0 ? num_topk : 1;
    const StashLayout l = stash_layout(requests, canvas_len, vocab, kq);
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    StashParams p{};
    p.logits = logits;
    p.row_stride = row_stride;
    p.logits_rows = logits_rows;
    p.vocab = static_cast<int32_t>(vocab);
    p.canvas_len = canvas_len;
    p.requests = requests;
    p.out_slots = out_slots;
    p.src = src;
    p.slots = slots;
    p.keep = keep;
    p.valid = valid;
    p.temps = temps;
    p.num_topk = num_topk;
    p.kq = kq;
    p.num_token_ids = num_token_ids;
    p.token_ids = token_ids;
    p.ids_stride = ids_stride;
    p.width = width;
    p.logits_mode = logits_mode ? 1 : 0;
    p.out_ids = out_ids;
    p.out_vals = out_logprobs;
    p.out_ranks = out_ranks;
    p.list = reinterpret_cast<int32_t*>(ws + l.list);
    p.map_row = reinterpret_cast<int32_t*>(ws + l.map_row);
    p.map_temp = reinterpret_cast<float*>(ws + l.map_temp);
    p.map_out = reinterpret_cast<int64_t*>(ws + l.map_out);
    p.map_req = reinterpret_cast<int32_t*>(ws + l.map_req);
    int32_t* top_ids = reinterpret_cast<int32_t*>(ws + l.top_ids);
    float* top_lp = reinterpret_cast<float*>(ws + l.top_lp);
    float* row_m = reinterpret_cast<float*>(ws + l.row_m);
    float* row_logs = reinterpret_cast<float*>(ws + l.row_logs);
    p.top_ids = top_ids;
    p.top_lp = top_lp;
    p.row_m = row_m;
    p.row_logs = row_logs;
    if (kq <= split_max_k()) {
        // the row kernels' list, header and RowTemps come from the list kernel
        const SplitPrepTargets tg =
            split_prep_targets(ws + l.split, requests * canvas_len, vocab, kq, 1);
        p.pass_list = tg.list;
        p.pass_header = tg.header;
        p.pass_rt = static_cast<rs::RowTemp*>(tg.row_temps);
    }

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t R = requests * canvas_len;
    stash_list<<<1, kListThreads, 0, st>>>(p);  // writes the list's count too
    if (cudaGetLastError() != cudaSuccess) return DRS_ERR_CUDA;
    const ExactTopkMap map{p.map_row, p.map_temp, row_m, row_logs};
    const int32_t* exact_list = p.list;
    if (kq <= split_max_k()) {
        // the one-read top-k over the listed rows; the rows it leaves (no
        // threshold, too many candidates) are on the hard-row list at the
        // start of its workspace
        RowCall c{};
        c.logits = logits;
        c.rows = R;
        c.vocab = vocab;
        c.row_stride = row_stride;
        c.canvas_len = 1;
        c.n_seeds = 1;
        c.probs_dtype = DRS_PROBS_NONE;
        c.k = kq;
        c.out_ids = top_ids;
        c.out_lp = top_lp;
        c.stats = false;
        c.map_row = p.map_row;
        c.map_temp = p.map_temp;
        c.map_count = p.list;
        c.out_m = row_m;
        c.out_logs = row_logs;
        c.prepared = true;
        const drs_status s = split_rows(c, ws + l.split, st);
        if (s != DRS_OK) return s;
        exact_list = reinterpret_cast<const int32_t*>(ws + l.split);
    }
    const drs_status s = exact_topk(logits, R, vocab, row_stride, 0, nullptr, 1, nullptr, exact_list,
                                    kq, top_ids, top_lp, ws + l.exact, st, &map);
    if (s != DRS_OK) return s;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((R + kWriteWarps - 1) / kWriteWarps));
    cfg.blockDim = dim3(kWriteWarps * 32);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, stash_write, p) == cudaSuccess ? DRS_OK : DRS_ERR_CUDA;
}
