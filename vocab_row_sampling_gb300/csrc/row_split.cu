// row_split.cu -- the row statistics of temperature-scaled logits (argmax,
// Gumbel-max sample, softmax entropy, optionally the softmax in bf16/fp16)
// and the top-k logprobs of the rows of converged slots, in two streaming
// passes over the logits (page "vllm.model_executor.models.
// diffusion_gemma_sampler": module docstring, sample_row_stats,
// sample_row_stats_reference, stash_converged_logprobs, _lp_topk_kernel).
//
// Layout of the work. A row of V fp32 logits is cut into tiles: 6144
// columns in pass 1, 8192 in pass 2. A CTA of 256 threads works on one tile
// at a time (slot i of thread t holds columns 4*(i*256+t)+0..3 of the tile,
// i < 6 or 8); the CTAs of a persistent grid take the tiles of the rows of a
// work list round robin.
// No CTA ever waits for another: the tiles of a row meet through records in
// global memory that a later kernel on the stream merges.
//
// Kernels, in stream order:
//   prep   the rows that pass 1 works on (all rows, or the rows of converged
//          slots in top-k-only calls) into a list, with each row's
//          temperature and its quotient constants.
//   pass 1 per tile, per warp: the warp max M_w of the scaled logits s = x /
//          Te (Te = max(T, 1e-10)) and the lowest column reaching it;
//          S_w = sum e^(s - M_w), W_w = sum e^(s - M_w) (s - M_w) (the online
//          max and sum of the page). While |M_w| < 256 the warp works on the
//          raw logits: the max is found among them, only the candidates for
//          the argmax are divided (exactly), and e^(s - M_w) = 2^(x log2(e) /
//          Te - c), c the rounded reference; warps with larger scaled values
//          divide every logit exactly first. The tile's record combines the
//          warps, with the Gumbel-max score of each warp's argmax element and
//          the warps' raw maxima.
//   merge  one warp per row (one CTA of 8 warps per row for rows of more
//          than 60 pass-1 tiles): max M, S, W (entropy log S - W / S), argmax, B =
//          the best of the warps' argmax scores, and the top-k threshold thr
//          = the k-th largest raw warp maximum (k distinct elements reach it,
//          so the row's top k all do); the row's record, and the list of rows
//          that pass 2 works on.
//   pass 2 per tile: the probabilities 2^(x log2(e) / Te - c2) (c2 the rounded
//          log2 of e^M S), rounded to nearest even; the pruned race against B
//          (an element can only win if 1 - u <= -log u <= e^(s - B): float4
//          groups whose largest e^(s - B) is below 2^-24 are dropped, the
//          others go on a per-warp list shared out one Philox call per lane,
//          and the few survivors are rescored exactly); the top-k candidates
//          x >= thr, keyed by (exact scaled value, lower column).
//   finish one warp per row: the sample (the best of the tiles' race winners
//          and B); the top k of the row's candidates by rank, logprob
//          s - M - log S. Rows whose candidates overflow the lists, or that
//          have no threshold, go on a device list for the exact top-k kernel.
//
// The passes stream their tiles through two shared-memory stages per CTA
// (three CTAs per SM) filled by bulk copies (TMA), the row's record riding
// along with each tile. Warps run freely: a warp waits for a stage's copy,
// works on the tile and counts itself out of the stage; the warp that
// counts out last finishes the tile (combines the warps' results) and
// refills the stage. No CTA-wide barrier in the loop.
//
// HBM traffic: every logit is read twice (once per pass) and every
// probability written once; the records are a few bytes per thousand
// logits. No fp64 arithmetic.
//
// A call can also pass a row map (the stash): its rows are then the entries
// of a device list, each read from a mapped logits row with a mapped
// temperature.
#include <algorithm>

#include "row_common.cuh"

namespace drs {
using namespace rs;
namespace {


// ------------------------------------------------------- tile pipeline

// Shared state of a CTA's pipeline. Tile n of the CTA is t_n = blockIdx.x +
// n * grid of its pass's tile space (list index * G + tile of the row); it
// goes through stage n % kStages. The ring `row`/`col` maps tile n (entry n
// % kMap) to its row and tile of the row, -1 past the end.
struct Pipe {
    uint64_t full[kStages];
    int count[kStages];
    int last_n[kStages];  // last tile issued into each stage
    int abort;
    int row[kMap];
    int col[kMap];
    int lrow[kMap];  // the logits row of `row` (differs under a row map)
};

// The tiles of a launch: [t_begin, t_end) of the list's tile space.
struct TileRange {
    int64_t t_begin, t_end;
};

// Map tiles first .. first + nfill - 1 (one per lane or thread).
__device__ __forceinline__ void map_tiles(Pipe& pp, const int32_t* list, const int32_t* map_row,
                                          TileRange tr, int G, int first, int nfill, int idx) {
    if (idx >= nfill) return;
    const int n = first + idx;
    const int64_t t = tr.t_begin + static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(n) * gridDim.x;
    int row = -1, c = 0, lrow = -1;
    if (t < tr.t_end) {
        const uint32_t li = static_cast<uint32_t>(t) / static_cast<uint32_t>(G);
        c = static_cast<int>(static_cast<uint32_t>(t) - li * static_cast<uint32_t>(G));
        row = list[li];
        lrow = map_row ? map_row[row] : row;
    }
    pp.row[n % kMap] = row;
    pp.col[n % kMap] = c;
    pp.lrow[n % kMap] = lrow;
}

// Issue tile n into its stage: the row's record (`rec_bytes` of `rec_table`)
// and the tile's whole float4s by bulk copy when rows start 16-byte aligned
// (else the warps read global memory themselves). Past the end: a plain
// arrival. COLS: the pass's tile width.
template <int COLS>
__device__ __forceinline__ void issue_tile(const SplitParams& p, Pipe& pp, int n, float4* stage,
                                           void* rec_dst, const void* rec_table, uint32_t rec_bytes,
                                           bool tma) {
    const int st = n % kStages;
    const int row = pp.row[n % kMap];
    pp.last_n[st] = n;
    if (p.fault && n == 0 && blockIdx.x == 0 && rec_bytes == sizeof(RowTemp)) {
        // the test hook: the stage never fills, its waits run out
        pp.last_n[st] = -1;
        return;
    }
    if (row < 0) {
        mbar_arrive(&pp.full[st]);
        return;
    }
    const int col0 = pp.col[n % kMap] * COLS;
    const int ncols = min(p.vocab - col0, COLS);
    const uint32_t bytes = tma ? static_cast<uint32_t>(ncols >> 2) * 16u : 0u;
    mbar_arrive_expect_tx(&pp.full[st], bytes + rec_bytes);
    tma_load_1d(rec_dst, static_cast<const unsigned char*>(rec_table) + static_cast<size_t>(row) * rec_bytes,
                rec_bytes, &pp.full[st]);
    if (bytes)
        tma_load_1d(stage, p.logits + static_cast<int64_t>(pp.lrow[n % kMap]) * p.row_stride + col0, bytes,
                    &pp.full[st]);
}

// The tiles of this launch: the list entries' tiles.
__device__ __forceinline__ TileRange launch_tiles(const SplitParams& p, int G) {
    return TileRange{static_cast<int64_t>(list_begin(p)) * G, static_cast<int64_t>(list_end(p)) * G};
}

// Pipeline start: barriers, the first kMap tiles mapped, the first kStages
// issued (the row record of stage s at recs + s * rec_stride). COLS: the
// pass's tile width; G: its tiles per row.
template <int COLS>
__device__ __forceinline__ void pipe_start(const SplitParams& p, Pipe& pp, const int32_t* list,
                                           TileRange tiles, int G, float4* stages, void* recs,
                                           size_t rec_stride, const void* rec_table,
                                           uint32_t rec_bytes, bool tma) {
    const int tid = threadIdx.x;
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&pp.full[s], 1);
            pp.count[s] = 0;
        }
        pp.abort = 0;
        fence_barrier_init();
    }
    map_tiles(pp, list, p.map_row, tiles, G, 0, kMap, tid);
    __syncthreads();
    if (tid == 0)
        for (int s = 0; s < kStages; ++s)
            issue_tile<COLS>(p, pp, s, stages + s * (COLS / 4), static_cast<unsigned char*>(recs) + s * rec_stride,
                             rec_table, rec_bytes, tma);
}

// The last warp out of tile n: refill its stage with tile n + kStages, and
// every 32 tiles map 32 more (over tiles that every warp is done with).
template <int COLS>
__device__ __forceinline__ void pipe_advance(const SplitParams& p, Pipe& pp, int n, const int32_t* list,
                                             TileRange tiles, int G, float4* stage, void* rec_dst,
                                             const void* rec_table, uint32_t rec_bytes, bool tma,
                                             int lane) {
    if (lane == 0) {
        fence_proxy_async_smem();
        issue_tile<COLS>(p, pp, n + kStages, stage, rec_dst, rec_table, rec_bytes, tma);
    }
    if ((n & 31) == 31) map_tiles(pp, list, p.map_row, tiles, G, n + 33, 32, lane);
}

// After the loop: if a wait ran out, copies still in flight land before the
// CTA's shared memory is released.
__device__ __forceinline__ void pipe_end(Pipe& pp) {
    __syncthreads();
    if (threadIdx.x == 0 && pp.abort)
        for (int s = 0; s < kStages; ++s)
            if (pp.last_n[s] >= 0)
                mbar_wait_bounded(&pp.full[s], static_cast<uint32_t>((pp.last_n[s] / kStages) & 1));
}

// A thread's float4 slots of the tile (-inf past the row's end): from the
// stage; the ragged last float4 and (without bulk copies) everything from
// global memory, stored into the stage as well, so that the stage always
// holds the whole tile.
template <int VEC>
__device__ __forceinline__ void read_tile(float4 (&v)[VEC], float4* stage, const float* tp,
                                          int ncols, int tid, bool tma) {
    if (tma && ncols == kSThreads * VEC * 4) {
#pragma unroll
        for (int i = 0; i < VEC; ++i) v[i] = stage[i * kSThreads + tid];
        return;
    }
    const int nfull4 = ncols >> 2;
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
        const int f = i * kSThreads + tid;
        float4 x = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        if (f < nfull4) {
            if (tma) {
                x = stage[f];
            } else {
                x = make_float4(__ldcs(tp + 4 * f), __ldcs(tp + 4 * f + 1), __ldcs(tp + 4 * f + 2),
                                __ldcs(tp + 4 * f + 3));
                stage[f] = x;
            }
        } else if (f == nfull4 && (ncols & 3)) {
            for (int q = 0; q < (ncols & 3); ++q) set_comp(x, q, __ldcs(tp + 4 * f + q));
            stage[f] = x;
        }
        v[i] = x;
    }
}

// ================================================================ prep

// The list of rows the passes work on, in row order, and each listed row's
// RowTemp. The order is fixed so that a call divides its list between the
// cluster kernel and the two passes the same way on every run (the two sum a
// row's exponentials in different orders). With statistics, every row is
// listed: the list is the identity. With a row map (the stash), the first
// *map_count entries when k > 0. Otherwise (top-k-only calls) the rows of
// kept slots: CTA 0 walks the rows 256 at a time and places each kept row
// after the kept rows before it (a block-wide count); the other CTAs write
// the RowTemps of their rows. The list header too: its length, and the
// hard-row count set to 0 (the kernels after it add to it).
__device__ __forceinline__ bool prep_row(const SplitParams& p, int64_t row) {
    if (row >= p.rows) return false;
    uint64_t slot = 0;
    bool kept;
    if (p.map_row) {
        kept = row < *p.map_count;  // every listed entry is kept
    } else {
        slot = slot_of(p, static_cast<uint64_t>(p.row0 + row));
        kept = p.keep == nullptr || p.keep[slot] != 0;
    }
    const bool work = (p.stats && !p.map_row) || (p.k > 0 && kept);
    if (work) {
        const float temp = p.map_row ? p.map_temp[row] : p.temps[slot];
        const ScaledQuotient q = ScaledQuotient::of(fmaxf(temp, kTempFloor));
        p.rt[row] = RowTemp{temp, q.t, q.y, q.mode};
    }
    return work;
}

__global__ void __launch_bounds__(256) split_prep(const __grid_constant__ SplitParams p) {
    const int64_t row = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (p.stats || p.map_row) {
        const int64_t n = p.map_row ? (p.k > 0 ? min(static_cast<int64_t>(*p.map_count), p.rows) : 0) : p.rows;
        if (prep_row(p, row) && row < n) p.list1[row] = static_cast<int32_t>(row);
        if (row == 0) {
            p.hard[0] = 0;  // the hard-row count, before pass 1
            p.hard[kCount1] = static_cast<int32_t>(n);
        }
        return;
    }
    if (blockIdx.x != 0) {
        prep_row(p, row);
        return;
    }
    __shared__ int wcount[8];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    int base = 0;
    for (int64_t r0 = 0; r0 < p.rows; r0 += 256) {
        const int64_t r = r0 + threadIdx.x;
        // rows of CTA 0's own block: their RowTemp too; later rows: the flag
        const bool work = r < 256 ? prep_row(p, r)
                                  : r < p.rows && p.k > 0 &&
                                        (p.keep == nullptr || p.keep[slot_of(p, static_cast<uint64_t>(p.row0 + r))] != 0);
        const uint32_t b = __ballot_sync(0xffffffffu, work);
        if (lane == 0) wcount[warp] = __popc(b);
        __syncthreads();
        int before = base, total = 0;
        for (int w = 0; w < 8; ++w) {
            before += w < warp ? wcount[w] : 0;
            total += wcount[w];
        }
        if (work) p.list1[before + __popc(b & lanemask_lt())] = static_cast<int32_t>(r);
        base += total;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        p.hard[0] = 0;  // the hard-row count, before pass 1
        p.hard[kCount1] = base;
    }
}

// ============================================================== pass 1


// A warp's S = sum 2^t and W = ln2 * sum 2^t t, t = x * lscale - cref, over
// the thread's slots; with CLAMP, t is kept finite (a -inf logit gives e = 0
// and e * t = 0 instead of NaN).
template <bool CLAMP, int VEC>
__device__ __forceinline__ void tile_sums(const float4 (&v)[VEC], float lscale, float cref,
                                          float& sw, float& ww) {
    float sa[4] = {0.0f, 0.0f, 0.0f, 0.0f}, wa[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float tq = fmaf(comp(v[i], q), lscale, -cref);
            if (CLAMP) tq = fmaxf(tq, -FLT_MAX);
            const float e = ex2_ftz(tq);
            sa[q] += e;
            wa[q] = fmaf(e, tq, wa[q]);
        }
    }
    sw = warp_sum_f((sa[0] + sa[1]) + (sa[2] + sa[3]));
    ww = warp_sum_f((wa[0] + wa[1]) + (wa[2] + wa[3])) * kLn2;
}

// One warp's share of a pass-1 tile: M_w's raw max and its lowest column,
// S_w and W_w relative to it.
__device__ __forceinline__ WarpPart p1_warp(const SplitParams& p, float4* stage, const ScaledQuotient& sq,
                                            int lrow, int col0, int ncols, int tid, int lane, bool stats,
                                            bool tma) {
    float4 v[kP1Vec4];
    read_tile(v, stage, p.logits + static_cast<int64_t>(lrow) * p.row_stride + col0, ncols, tid, tma);

    // max of the raw logits (division by Te > 0 keeps the order)
    float m4[kP1Vec4];
    float mt = -INFINITY;
#pragma unroll
    for (int i = 0; i < kP1Vec4; ++i) {
        m4[i] = max4f(v[i]);
        mt = fmaxf(mt, m4[i]);
    }
    const float mxw = warp_max_f(mt);
    // the warp works on the raw logits while |M_w| < 256 for sure:
    // |mxw * RN(1/Te)| < 255 bounds the exact quotient M_w (computed
    // once per tile for all warps by the warp that finishes it)
    const bool raw = fabsf(mxw * sq.y) < kRawLimit - 1.0f;

    // the lowest column holding mxw (its exact quotient is M_w): the
    // warp's Gumbel-max candidate, and the argmax unless a lower
    // logit has the same exact quotient (pass 2 looks for those).
    // The lane's first slot reaching mxw is read again from the stage.
    int arg_t = INT_MAX;
    if (stats && mt == mxw && mxw != -INFINITY) {
        int i0 = 0;
#pragma unroll
        for (int i = kP1Vec4 - 1; i >= 0; --i)
            if (m4[i] == mxw) i0 = i;
        const int f = i0 * kSThreads + tid;
        const float4 x4 = stage[f];
        const int q = x4.x == mxw ? 0 : x4.y == mxw ? 1 : x4.z == mxw ? 2 : 3;
        arg_t = col0 + 4 * f + q;
    }
    const int aw = stats ? warp_min_nonneg(arg_t) : INT_MAX;

    // t = (s - M_w) log2(e): raw x * log2(e)/Te - c, c = RN(mxw *
    // log2(e)/Te), else (s - M_w) * log2(e). Terms below 2^-126 of
    // S >= 1 are flushed. A -inf logit (e = 0, t = -inf) makes W NaN:
    // such warps sum again with t clamped to a finite value.
    float lscale, cref;
    if (raw) {
        lscale = kLog2e * sq.y;
        cref = mxw * lscale;
    } else {
        // (logits whose exponential is 0 anyway are not divided; a slot
        // none of the warp's lanes needs is skipped)
        const float mw = sq.exact(mxw);
        const FarBelow far(mxw, kLog2e * sq.y);
#pragma unroll
        for (int i = 0; i < kP1Vec4; ++i) {
            const bool f0 = far(v[i].x), f1 = far(v[i].y), f2 = far(v[i].z), f3 = far(v[i].w);
            if (__any_sync(0xffffffffu, !(f0 && f1 && f2 && f3))) {
                v[i].x = f0 ? kFarStandIn : sq.exact(v[i].x) - mw;
                v[i].y = f1 ? kFarStandIn : sq.exact(v[i].y) - mw;
                v[i].z = f2 ? kFarStandIn : sq.exact(v[i].z) - mw;
                v[i].w = f3 ? kFarStandIn : sq.exact(v[i].w) - mw;
            } else {
                v[i] = make_float4(kFarStandIn, kFarStandIn, kFarStandIn, kFarStandIn);
            }
        }
        lscale = kLog2e;
        cref = 0.0f;
    }
    float sw = 0.0f, ww = 0.0f;  // a warp of -inf only: nothing to sum
    if (mxw != -INFINITY) {
        tile_sums<false, kP1Vec4>(v, lscale, cref, sw, ww);
        if (isnan(ww)) tile_sums<true, kP1Vec4>(v, lscale, cref, sw, ww);
    }
    return WarpPart{0.0f, sw, ww, mxw, aw};
}

// The record of a pass-1 tile from its warps' parts (one lane each).
__device__ __forceinline__ void p1_combine(const SplitParams& p, const WarpPart (&parts)[kSWarps],
                                           const ScaledQuotient& sq, int64_t t, int col0, int ncols,
                                           int lane) {
    const bool hv = lane < kSWarps;
    WarpPart wp = hv ? parts[lane] : WarpPart{-INFINITY, 0.0f, 0.0f, -INFINITY, INT_MAX};
    wp.m = wp.xmax == -INFINITY ? -INFINITY : sq.exact(wp.xmax);  // M_w of each warp
    const float mc = warp_max_f(wp.m);
    float s_l = 0.0f, w_l = 0.0f;
    if (wp.m != -INFINITY) {
        const float dm = wp.m - mc;
        const float f = ex2_approx(dm * kLog2e);
        s_l = f * wp.s;
        w_l = f * fmaf(dm, wp.s, wp.w);
    }
    const float s_c = warp_sum_f(s_l);
    const float w_c = warp_sum_f(w_l);
    const float xm = warp_max_f(wp.xmax);
    const int a_c = xm == -INFINITY ? col0 : warp_min_nonneg(wp.xmax == xm ? wp.arg : INT_MAX);
    TileStats* dst = p.ts + t;
    if (hv) {
        dst->wmax[lane] = lane * 128 < ncols ? ord32(wp.xmax) : 0u;
        dst->wcol[lane] = wp.arg;
    }
    if (lane == 0) {
        dst->m = mc;
        dst->s = s_c;
        dst->w = w_c;
        dst->arg = a_c;
        dst->xmax = xm;
    }
}

// Pass 1, the merge, pass 2 and the finish are launched as programmatic
// dependents: each may be scheduled while its predecessor drains, waits for
// it to complete (griddepcontrol.wait, a no-op without the launch attribute)
// before anything else, and lets its own dependent launch once a CTA's work
// is done.
__global__ void __launch_bounds__(kSThreads, DRS_P1_MINB) split_pass1(const __grid_constant__ SplitParams p) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    extern __shared__ __align__(128) unsigned char smem[];
    float4* stages = reinterpret_cast<float4*>(smem);
    __shared__ Pipe pp;
    __shared__ RowTemp rts[kStages];
    __shared__ WarpPart parts[2][kStages][kSWarps];
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const bool stats = p.stats != 0;
    const bool tma = p.vec != 0;
    const TileRange tiles = launch_tiles(p, p.tiles1);
    pipe_start<kP1Cols>(p, pp, p.list1, tiles, p.tiles1, stages, rts, sizeof(RowTemp), p.rt, sizeof(RowTemp),
                        tma);
    for (int n = 0;; ++n) {
        const int st = n % kStages;
        const int par = (n / kStages) & 1;
        float4* stage = stages + st * (kP1Cols / 4);
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&pp.full[st], static_cast<uint32_t>(par)))) {
            if (lane == 0) {
                pp.abort = 1;
                raise_device_error(p.err, 1);
            }
            break;
        }
        const int row = pp.row[n % kMap];
        if (row < 0) break;
        const int64_t t = tiles.t_begin + static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(n) * gridDim.x;
        const int col0 = pp.col[n % kMap] * kP1Cols;
        const int ncols = min(p.vocab - col0, kP1Cols);
        ScaledQuotient sq;
        sq.t = rts[st].qt;
        sq.y = rts[st].qy;
        sq.mode = rts[st].qmode;
        const WarpPart wp = p1_warp(p, stage, sq, pp.lrow[n % kMap], col0, ncols, tid, lane, stats, tma);
        if (lane == 0) parts[par][st][warp] = wp;
        if (!release_stage(&pp.count[st], lane)) continue;

        // the last warp out: refill the stage, then the tile's record (the
        // warps combined, one lane each)
        pipe_advance<kP1Cols>(p, pp, n, p.list1, tiles, p.tiles1, stage, &rts[st], p.rt, sizeof(RowTemp), tma,
                              lane);
        p1_combine(p, parts[par][st], sq, t, col0, ncols, lane);
    }
    asm volatile("griddepcontrol.launch_dependents;");
    pipe_end(pp);
}

// ============================================================== merge

constexpr int kRowWarps = 8;  // rows per CTA of the merge and finish kernels

// Shared memory of a merge CTA whose W warps share one row (W > 1): one slot
// per warp for each cross-warp reduction, and each warp's k largest warp
// maxima.
template <int W>
struct MergeShared {
    float f[4][W];
    int i[W];
    float bs[W];
    int bc[W];
    uint32_t lists[W][kSplitMaxK];
    uint32_t kth;
};

// A warp-reduced value combined over the W warps of a row (W = 1: itself).
// Every thread of the CTA calls it; slot `red` is free again on return.
template <int W, typename T, typename Op>
__device__ __forceinline__ T across_warps(T v, T* red, int lane, int warp, Op op) {
    if constexpr (W == 1) {
        return v;
    } else {
        if (lane == 0) red[warp] = v;
        __syncthreads();
        T r = red[0];
#pragma unroll
        for (int i = 1; i < W; ++i) r = op(r, red[i]);
        __syncthreads();
        return r;
    }
}

// The merge of list entry li by W warps (thread r of 32 W): the row's M, S,
// W, argmax, the warps' Gumbel-max candidates scored per seed (B), the top-k
// threshold, the row record for pass 2, the entropy; rows without a
// threshold go on the hard-row list. NU: warp maxima per thread.
template <int NU, int W>
__device__ __forceinline__ void merge_row(const SplitParams& p, int64_t li, int r, MergeShared<W>* sh) {
    const int lane = r & 31;
    const int warp = r >> 5;
    constexpr int kStride = 32 * W;
    const int64_t row = p.list1[li];
    const bool kept =
        p.map_row || p.keep == nullptr || p.keep[slot_of(p, static_cast<uint64_t>(p.row0 + row))] != 0;
    const RowTemp rt = p.rt[row];
    const float temp = rt.temp;
    const int G = p.tiles1;  // the row's pass-1 tile records
    const TileStats* tr = p.ts + li * G;
    float m = -INFINITY, s = 0.0f, w = 0.0f, xm = -INFINITY;
    int arg = INT_MAX;
    for (int c = r; c < G; c += kStride) {
        const TileStats ti = tr[c];
        // the lowest column holding the raw max (-inf rows: the first)
        arg = ti.xmax > xm ? ti.arg : (ti.xmax == xm ? min(arg, ti.arg) : arg);
        xm = fmaxf(xm, ti.xmax);
        if (ti.m != -INFINITY) {
            if (m == -INFINITY) {
                m = ti.m;
                s = ti.s;
                w = ti.w;
            } else {
                const float nm = fmaxf(m, ti.m);
                const float d1 = m - nm, d2 = ti.m - nm;
                const float f1 = ex2_approx(d1 * kLog2e), f2 = ex2_approx(d2 * kLog2e);
                w = f1 * fmaf(d1, s, w) + f2 * fmaf(d2, ti.s, ti.w);
                s = f1 * s + f2 * ti.s;
                m = nm;
            }
        }
    }
    auto fmax_op = [](float a, float b) { return fmaxf(a, b); };
    auto fsum_op = [](float a, float b) { return a + b; };
    auto imin_op = [](int a, int b) { return min(a, b); };
    float* redf0 = W > 1 ? sh->f[0] : nullptr;
    float* redf1 = W > 1 ? sh->f[1] : nullptr;
    float* redf2 = W > 1 ? sh->f[2] : nullptr;
    float* redf3 = W > 1 ? sh->f[3] : nullptr;
    int* redi = W > 1 ? sh->i : nullptr;
    const float big_m = across_warps<W>(warp_max_f(m), redf0, lane, warp, fmax_op);
    float s_l = 0.0f, w_l = 0.0f;
    if (m != -INFINITY) {
        const float dm = m - big_m;
        const float f = ex2_approx(dm * kLog2e);
        s_l = f * s;
        w_l = f * fmaf(dm, s, w);
    }
    const float s_tot = across_warps<W>(warp_sum_f(s_l), redf1, lane, warp, fsum_op);
    const float w_tot = across_warps<W>(warp_sum_f(w_l), redf2, lane, warp, fsum_op);
    const float mraw = across_warps<W>(warp_max_f(xm), redf3, lane, warp, fmax_op);
    const int arg_row = across_warps<W>(warp_min_nonneg(xm == mraw ? arg : INT_MAX), redi, lane, warp, imin_op);

    const bool topk = p.k > 0 && kept;
    float thr = -INFINITY;
    bool hard = false;
    if (topk) {
        // the k-th largest of the row's warp maxima (absent warps are 0,
        // below every value): k rounds of a warp max, each removing one
        // occurrence; with W warps, each warp's k largest, then the k-th
        // largest of their union (a merge of W sorted lists)
        uint32_t o[NU];
#pragma unroll
        for (int u = 0; u < NU; ++u) {
            const int jx = r + kStride * u;
            o[u] = jx < kSWarps * G ? tr[jx / kSWarps].wmax[jx % kSWarps] : 0u;
        }
        uint32_t kth = 0;
        for (int rd = 0; rd < p.k; ++rd) {
            uint32_t lm = 0;
#pragma unroll
            for (int u = 0; u < NU; ++u) lm = max(lm, o[u]);
            uint32_t top;
            asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(top) : "r"(lm));
            kth = top;
            if (W > 1 && lane == 0) sh->lists[warp][rd] = top;
            const uint32_t holders = __ballot_sync(0xffffffffu, lm == top);
            if (lane == __ffs(holders) - 1) {
                bool done = false;
#pragma unroll
                for (int u = 0; u < NU; ++u)
                    if (!done && o[u] == top) {
                        o[u] = 0;
                        done = true;
                    }
            }
        }
        if constexpr (W > 1) {
            // lane j < W of warp 0 holds the head of warp j's list; each
            // round takes the largest head
            __syncthreads();
            if (warp == 0) {
                int at = 0;
                uint32_t head = lane < W ? sh->lists[lane][0] : 0u;
                for (int rd = 0; rd < p.k; ++rd) {
                    uint32_t top;
                    asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(top) : "r"(head));
                    kth = top;
                    const uint32_t holders = __ballot_sync(0xffffffffu, lane < W && head == top);
                    if (lane == __ffs(holders) - 1) {
                        ++at;
                        head = at < p.k ? sh->lists[lane][at] : 0u;
                    }
                }
                if (lane == 0) sh->kth = kth;
            }
            __syncthreads();
            kth = sh->kth;
        }
        // absent, or -inf: no threshold, the exact kernel takes the row.
        // Lowered by Te ulp(s): a logit below thr whose exact quotient
        // equals thr's is a candidate too (equal values rank by column).
        if (kth > kOrdNegInf) {
            const float x = unord32(kth);
            thr = x - fmaxf(fabsf(x) * 0x1p-20f, rt.qt * 0x1p-140f);
        } else {
            hard = true;
        }
    }

    // B per seed: the best Gumbel-max score of the warps' candidates (the
    // lowest column holding each warp's raw max, whose exact quotient is
    // M_w)
    const bool noisy = p.stats && temp > 0.0f && big_m != -INFINITY;
    const float ls = kLog2e * rt.qy;
    const float c0 = mraw * ls;
    unsigned char* entry = p.rr + row * p.rec_bytes;
    for (int sd = 0; sd < p.n_seeds; ++sd) {
        float b = -INFINITY;
        int bc = INT_MAX;
        if (noisy) {
            const uint64_t grow = static_cast<uint64_t>(p.row0 + row);
            const ScaledQuotient sq{rt.qt, rt.qy, rt.qmode};
            for (int jx = r; jx < kSWarps * G; jx += kStride) {
                const int col = tr[jx / kSWarps].wcol[jx % kSWarps];
                if (col == INT_MAX) continue;
                const float mw = sq.exact(unord32(tr[jx / kSWarps].wmax[jx % kSWarps]));
                const uint4 nw = noise_group(p.rk[sd], grow, static_cast<uint32_t>(col >> 2));
                const float sc = mw + gumbel_of_bits(word_of(nw, col & 3));
                if (beats(sc, col, b, bc)) {
                    b = sc;
                    bc = col;
                }
            }
        }
        warp_best(b, bc);
        if constexpr (W > 1) {
            if (lane == 0) {
                sh->bs[warp] = b;
                sh->bc[warp] = bc;
            }
            __syncthreads();
            for (int j = 0; j < W; ++j)
                if (beats(sh->bs[j], sh->bc[j], b, bc)) {
                    b = sh->bs[j];
                    bc = sh->bc[j];
                }
            __syncthreads();
        }
        if (r == 0)
            reinterpret_cast<SeedRec*>(entry + sizeof(RowRecord))[sd] =
                SeedRec{b, (c0 + (b - big_m) * kLog2e) - kRaceSlack, bc, 0};
    }

    if (r == 0) {
        RowRecord rec{};
        rec.M = big_m;
        rec.log2s = s_tot > 0.0f ? log2f(s_tot) : 0.0f;
        rec.lns = rec.log2s * kLn2;
        rec.ls = ls;
        const bool raw = !(fabsf(big_m) >= kRawLimit);
        rec.c2 = c0 + rec.log2s;
        rec.thr = thr;
        rec.arg = arg_row;
        rec.cthr = mraw - fmaxf(fabsf(mraw) * 0x1p-20f, rt.qt * 0x1p-140f);
        rec.qt = rt.qt;
        rec.qy = rt.qy;
        rec.qmode = rt.qmode;
        rec.flags = (noisy ? kFNoisy : 0) | (topk && !hard ? kFTopk : 0) | (raw ? kFRaw : 0);
        *reinterpret_cast<RowRecord*>(entry) = rec;
        if (p.stats) p.entropy[row] = s_tot > 0.0f ? logf(s_tot) - w_tot / s_tot : 0.0f;
        if (p.out_m) {
            p.out_m[row] = big_m;
            p.out_logs[row] = rec.lns;
        }
        if (hard) {
            const int idx = atomicAdd(p.hard, 1);
            p.hard[kHardOffset + idx] = static_cast<int32_t>(row);
        }
    }
}

// W = 1: a row per warp, kRowWarps rows per CTA; W = kRowWarps: a row per
// CTA (long rows: the row's serial work split W ways)
template <int NU, int W>
__global__ void __launch_bounds__(kRowWarps * 32) split_merge(const __grid_constant__ SplitParams p) {
    static_assert(W == 1 || W == kRowWarps, "a merge CTA holds kRowWarps rows or one row");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if constexpr (W == 1) {
        const int64_t li = list_begin(p) + static_cast<int64_t>(blockIdx.x) * kRowWarps + (threadIdx.x >> 5);
        if (li >= list_end(p)) return;
        merge_row<NU, 1>(p, li, threadIdx.x & 31, nullptr);
    } else {
        __shared__ MergeShared<W> sh;
        const int64_t li = list_begin(p) + static_cast<int64_t>(blockIdx.x);
        if (li >= list_end(p)) return;  // the whole CTA
        merge_row<NU, W>(p, li, threadIdx.x, &sh);
    }
    asm volatile("griddepcontrol.launch_dependents;");
}

// ============================================================== pass 2

// The probabilities of a whole tile with aligned rows, no per-slot checks.
// FTZ: by the exponential that flushes subnormal results (one instruction),
// for threads none of whose probabilities is subnormal in fp32.
template <bool BF16, bool RAW, bool FTZ>
__device__ __forceinline__ void store_tile_probs(const float4 (&v)[kSVec4], const RowRecord& rec,
                                                 const ScaledQuotient& sq, uint16_t* prow, int tid) {
    const float ls = rec.ls, c2 = rec.c2, big_m = rec.M, l2s = rec.log2s;
    const FarBelow far(rec.cthr, ls);  // exact rows: cthr is at most the raw max
#pragma unroll
    for (int i = 0; i < kSVec4; ++i) {
        const int f = i * kSThreads + tid;
        float pr[4];
        // exact rows: a slot none of the warp's lanes needs is not divided
        const bool skip = !RAW && !__any_sync(0xffffffffu, !(far(v[i].x) && far(v[i].y) && far(v[i].z) &&
                                                             far(v[i].w)));
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float x = comp(v[i], q);
            const float tq = RAW              ? fmaf(x, ls, -c2)
                             : skip || far(x) ? kFarStandIn
                                              : fmaf(sq.exact(x) - big_m, kLog2e, -l2s);
            pr[q] = FTZ ? ex2_ftz(tq) : ex2_approx(tq);
        }
        __stcs(reinterpret_cast<uint2*>(prow + 4 * f),
               make_uint2(pack2<BF16>(pr[0], pr[1]), pack2<BF16>(pr[2], pr[3])));
    }
}

// Probabilities 2^t of a tile, t = x ls - c2 (raw rows) or (s - M) log2(e) -
// log2 S, subnormal results kept (bf16 can hold some); -inf logits give 0.
template <bool BF16, bool RAW>
__device__ __forceinline__ void write_probs(const float4 (&v)[kSVec4], const RowRecord& rec,
                                            const ScaledQuotient& sq, uint16_t* prow, bool vec,
                                            int ncols, int tid) {
    const float ls = rec.ls, c2 = rec.c2, big_m = rec.M, l2s = rec.log2s;
    // a whole tile with aligned rows: no per-slot checks (measured 6% of
    // pass 2 against the same loop with the checks)
    if (vec && ncols == kTileCols) {
        // fp16 holds nothing below 2^-25, so flushing fp32 subnormals
        // changes no fp16 code; for bf16 the thread's smallest logit tells
        // whether any of its probabilities is below 2^-126 (a NaN is
        // skipped by min; -inf gives t = -inf and the exact form)
        bool ftz = !BF16;
        if (BF16) {
            float xmin = min3(v[0].x, v[0].y, fminf(v[0].z, v[0].w));
#pragma unroll
            for (int i = 1; i < kSVec4; ++i) xmin = min3(xmin, min3(v[i].x, v[i].y, v[i].z), v[i].w);
            const float tmin = RAW ? fmaf(xmin, ls, -c2) : fmaf(sq.exact(xmin) - big_m, kLog2e, -l2s);
            ftz = tmin >= -126.0f;
        }
        if (ftz) store_tile_probs<BF16, RAW, true>(v, rec, sq, prow, tid);
        else store_tile_probs<BF16, RAW, false>(v, rec, sq, prow, tid);
        return;
    }
    // ragged tiles and rows without aligned 8-byte stores
#pragma unroll
    for (int i = 0; i < kSVec4; ++i) {
        const int f = i * kSThreads + tid;
        if (4 * f >= ncols) continue;
        float pr[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float x = comp(v[i], q);
            const float tq = RAW                              ? fmaf(x, ls, -c2)
                             : FarBelow(rec.cthr, ls)(x) ? kFarStandIn
                                                              : fmaf(sq.exact(x) - big_m, kLog2e, -l2s);
            pr[q] = ex2_approx(tq);
        }
        const uint32_t lo = pack2<BF16>(pr[0], pr[1]);
        const uint32_t hi = pack2<BF16>(pr[2], pr[3]);
        if (vec && 4 * f + 4 <= ncols) {
            __stcs(reinterpret_cast<uint2*>(prow + 4 * f), make_uint2(lo, hi));
        } else {
            const uint16_t code[4] = {static_cast<uint16_t>(lo), static_cast<uint16_t>(lo >> 16),
                                      static_cast<uint16_t>(hi), static_cast<uint16_t>(hi >> 16)};
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (4 * f + q < ncols) prow[4 * f + q] = code[q];
        }
    }
}

template <bool BF16>
__device__ __forceinline__ void probs_of_tile(const float4 (&v)[kSVec4], const RowRecord& rec,
                                              const ScaledQuotient& sq, uint16_t* prow, bool vec,
                                              int ncols, int tid) {
    if (rec.M == -INFINITY) {
        // a row that is -inf everywhere: NaN
        const uint16_t code = static_cast<uint16_t>(pack2<BF16>(NAN, NAN));
        for (int cidx = tid; cidx < ncols; cidx += kSThreads) prow[cidx] = code;
    } else if (rec.flags & kFRaw) {
        write_probs<BF16, true>(v, rec, sq, prow, vec, ncols, tid);
    } else {
        write_probs<BF16, false>(v, rec, sq, prow, vec, ncols, tid);
    }
}


// Shared memory of the pass-2 tile work: the race lists of the warps, and
// per tile in flight (parity of the tile's round, stage) the warps' race
// winners per seed, argmax ties and the tile's candidate count.
template <bool MULTI>
struct P2Shared {
    static constexpr int kSeedSlots = MULTI ? kMaxSeeds : 1;
    uint16_t race_at[kSWarps][kSVec4 * 32];
    float best_s[2][kStages][kSeedSlots][kSWarps];
    int best_c[2][kStages][kSeedSlots][kSWarps];
    int best_a[2][kStages][kSWarps];
    int tile_nk[2][kStages];
};

// One warp's share of a pass-2 tile (the row entry at `entry`: RowRecord,
// then one SeedRec per seed). Returns whether the row collects top-k
// candidates. MULTI: several noise seeds (a race per seed); else one, its
// round keys read as constants.
template <bool MULTI>
__device__ __forceinline__ bool p2_warp(const SplitParams& p, P2Shared<MULTI>& sh, float4* stage,
                                        const unsigned char* entry, int row, int lrow, int64_t t, int col0,
                                        int ncols, int st, int par, int tid, int lane, int warp,
                                        bool stats, bool probs, bool tma) {
    const RowRecord& rec = *reinterpret_cast<const RowRecord*>(entry);
    const SeedRec* seeds = reinterpret_cast<const SeedRec*>(entry + sizeof(RowRecord));
    const int flags = rec.flags;
    const bool noisy = (flags & kFNoisy) != 0;
    const bool topk = (flags & kFTopk) != 0;
    // (a row of a top-k-only call without a threshold, which the exact
    // kernel takes, runs through here with nothing to produce: it is
    // rare, and a branch around the block slowed every tile)
    {
        const uint64_t grow = static_cast<uint64_t>(p.row0 + row);
        ScaledQuotient sq;
        sq.t = rec.qt;
        sq.y = rec.qy;
        sq.mode = rec.qmode;
        float4 v[kSVec4];
        read_tile(v, stage, p.logits + static_cast<int64_t>(lrow) * p.row_stride + col0, ncols, tid, tma);

        if (probs) {
            uint16_t* prow = static_cast<uint16_t*>(p.probs) + static_cast<int64_t>(row) * p.probs_row_stride + col0;
            if (p.probs_dtype == 1) probs_of_tile<true>(v, rec, sq, prow, p.probs_vec != 0, ncols, tid);
            else probs_of_tile<false>(v, rec, sq, prow, p.probs_vec != 0, ncols, tid);
        }

        float m4[kSVec4];
#pragma unroll
        for (int i = 0; i < kSVec4; ++i) m4[i] = max4f(v[i]);
        // the thread's max: most threads hold nothing that reaches the
        // argmax or top-k bounds and skip both per-slot tests
        float mthr = m4[0];
#pragma unroll
        for (int i = 1; i < kSVec4; ++i) mthr = fmaxf(mthr, m4[i]);

        // argmax: logits below the raw max whose exact quotient is M
        // (rare: the float4s reaching the bound are read again from the
        // stage); the lowest column of the thread, then of the warp
        int acand = INT_MAX;
        if (stats && rec.M != -INFINITY) {
            const float cthr = rec.cthr;
            uint32_t am = 0;
            if (mthr >= cthr) {
#pragma unroll
                for (int i = 0; i < kSVec4; ++i) am |= (m4[i] >= cthr ? 1u : 0u) << i;
            }
#pragma unroll 1
            while (am && acand == INT_MAX) {
                const int f = (__ffs(am) - 1) * kSThreads + tid;
                am &= am - 1;
                const float4 x4 = stage[f];
#pragma unroll 1
                for (int q = 0; q < 4; ++q) {
                    const float x = comp(x4, q);
                    if (4 * f + q < ncols && x >= cthr && sq.exact(x) == rec.M) {
                        acand = col0 + 4 * f + q;
                        break;
                    }
                }
            }
            acand = warp_min_nonneg(acand);
        }

        // the race
        const bool rawr = (flags & kFRaw) != 0;
        if constexpr (!MULTI) {
        const int nsd = 1;
        for (int sd = 0; sd < nsd; ++sd) {
        const SeedRec sr = seeds[sd];
        const PhiloxRoundKeys& rk = MULTI ? p.rk[sd] : p.rk[0];
        float wb = sr.B;
        int wc = sr.bcol;
        if (noisy) {
            // groups whose largest e^(s - B) reaches 2^-24, listed
            // warp-wide by their float4 index in the stage
            uint32_t pass = 0;
            if (rawr) {
                const float ls = rec.ls, cB = sr.cB;
#pragma unroll
                for (int i = 0; i < kSVec4; ++i)
                    if (fmaf(m4[i], ls, -cB) >= -24.0f) pass |= 1u << i;
            } else {
#pragma unroll
                for (int i = 0; i < kSVec4; ++i)
                    if (fmaf(sq.exact(m4[i]) - sr.B, kLog2e, kRaceSlack) >= -24.0f) pass |= 1u << i;
            }
            const uint32_t lt = lanemask_lt();
            int total = 0;
#pragma unroll
            for (int i = 0; i < kSVec4; ++i) {
                const bool on = (pass >> i) & 1u;
                const uint32_t bl = __ballot_sync(0xffffffffu, on);
                if (on) sh.race_at[warp][total + __popc(bl & lt)] = static_cast<uint16_t>(i * kSThreads + tid);
                total += __popc(bl);
            }
            __syncwarp();
            // each listed group: its noise, then the group's largest e
            // against its largest word (one 2^x); the elements one by
            // one only when that passes
            for (int m = lane; m < total; m += 32) {
                const int f = sh.race_at[warp][m];
                const float4 x4 = stage[f];
                const int c4 = col0 + 4 * f;
                const uint4 nw = noise_group(rk, grow, static_cast<uint32_t>(c4 >> 2));
                const uint32_t wmax = max(max(nw.x, nw.y), max(nw.z, nw.w));
                const float mx = max4f(x4);
                const float emax = rawr ? ex2_ftz(fmaf(mx, rec.ls, -sr.cB))
                                        : ex2_ftz(fmaf(sq.exact(mx) - sr.B, kLog2e, kRaceSlack));
                if (one_minus_u_lower(wmax) <= emax) {
                    const float4 e = race_e(x4, rawr, rec.ls, sr, sq);
                    uint32_t bits = 0;
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (one_minus_u_lower(word_of(nw, q)) <= comp(e, q)) bits |= 1u << q;
                    if (bits) {
                        const Best b2 = race_rescore(bits, x4, nw, c4, sr.bcol, sq, Best{wb, wc});
                        wb = b2.s;
                        wc = b2.c;
                    }
                }
            }
            warp_best(wb, wc);
            if (MULTI) __syncwarp();  // the list is rewritten for the next seed
        }
        if (lane == 0) {
            sh.best_s[par][st][sd][warp] = wb;
            sh.best_c[par][st][sd][warp] = wc;
        }
        }
        } else {
        // several seeds: one list of the groups that some seed can still use
        // (the bound of the seed with the smallest cB, or B: the bound falls
        // with both), each listed group then raced for every seed in turn
        // (its float4 read once; each seed's noise drawn without a branch
        // before it, so the chains of consecutive seeds overlap, and a seed
        // whose own bound drops the group only fails the test)
        const int nsd = p.n_seeds;
        float wbs[kMaxSeeds];
        int wcs[kMaxSeeds];
#pragma unroll
        for (int sd = 0; sd < kMaxSeeds; ++sd) {
            wbs[sd] = sd < nsd ? seeds[sd].B : -INFINITY;
            wcs[sd] = sd < nsd ? seeds[sd].bcol : INT_MAX;
        }
        if (noisy) {
            float c_lo = INFINITY, b_lo = INFINITY;
            for (int sd = 0; sd < nsd; ++sd) {
                c_lo = fminf(c_lo, seeds[sd].cB);
                b_lo = fminf(b_lo, seeds[sd].B);
            }
            uint32_t pass = 0;
            if (rawr) {
                const float ls = rec.ls;
#pragma unroll
                for (int i = 0; i < kSVec4; ++i)
                    if (fmaf(m4[i], ls, -c_lo) >= -24.0f) pass |= 1u << i;
            } else {
#pragma unroll
                for (int i = 0; i < kSVec4; ++i)
                    if (fmaf(sq.exact(m4[i]) - b_lo, kLog2e, kRaceSlack) >= -24.0f) pass |= 1u << i;
            }
            const uint32_t lt = lanemask_lt();
            int total = 0;
#pragma unroll
            for (int i = 0; i < kSVec4; ++i) {
                const bool on = (pass >> i) & 1u;
                const uint32_t bl = __ballot_sync(0xffffffffu, on);
                if (on) sh.race_at[warp][total + __popc(bl & lt)] = static_cast<uint16_t>(i * kSThreads + tid);
                total += __popc(bl);
            }
            __syncwarp();
            for (int m = lane; m < total; m += 32) {
                const int f = sh.race_at[warp][m];
                const float4 x4 = stage[f];
                const int c4 = col0 + 4 * f;
                const float mx = max4f(x4);
                const float ex = rawr ? 0.0f : sq.exact(mx);
#pragma unroll
                for (int sd = 0; sd < kMaxSeeds; ++sd) {
                    if (sd >= nsd) break;
                    const SeedRec& sr = seeds[sd];
                    const float t = rawr ? fmaf(mx, rec.ls, -sr.cB) : fmaf(ex - sr.B, kLog2e, kRaceSlack);
                    const uint4 nw = noise_group(p.rk[sd], grow, static_cast<uint32_t>(c4 >> 2));
                    const uint32_t wmax = max(max(nw.x, nw.y), max(nw.z, nw.w));
                    if (t >= -24.0f && one_minus_u_lower(wmax) <= ex2_ftz(t)) {
                        const float4 e = race_e(x4, rawr, rec.ls, sr, sq);
                        uint32_t bits = 0;
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            if (one_minus_u_lower(word_of(nw, q)) <= comp(e, q)) bits |= 1u << q;
                        if (bits) {
                            const Best b2 = race_rescore(bits, x4, nw, c4, sr.bcol, sq, Best{wbs[sd], wcs[sd]});
                            wbs[sd] = b2.s;
                            wcs[sd] = b2.c;
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int sd = 0; sd < kMaxSeeds; ++sd) {
            if (sd >= nsd) break;
            float wb = wbs[sd];
            int wc = wcs[sd];
            warp_best(wb, wc);
            if (lane == 0) {
                sh.best_s[par][st][sd][warp] = wb;
                sh.best_c[par][st][sd][warp] = wc;
            }
        }
        }

        if (topk && mthr >= rec.thr) {
            // candidates x >= thr (rare: the slots reaching it)
            const float thr = rec.thr;
            uint32_t km = 0;
#pragma unroll
            for (int i = 0; i < kSVec4; ++i) km |= (m4[i] >= thr ? 1u : 0u) << i;
            if (km)
                topk_collect(km, stage, tid, col0, ncols, thr, sq, &sh.tile_nk[par][st],
                             p.keys + t * kTileKeys);
        }
        if (lane == 0) sh.best_a[par][st][warp] = acand;
    }
    return topk;
}

// The last warp out of a pass-2 tile: the tile's records (race winner per
// seed, candidate count, argmax tie).
template <bool MULTI>
__device__ __forceinline__ void p2_combine(const SplitParams& p, P2Shared<MULTI>& sh, int64_t t, int st,
                                           int par, bool stats, bool topk, int lane) {
    if (stats || topk) {
        const int nsd = MULTI ? p.n_seeds : 1;
        for (int sd = 0; sd < nsd; ++sd) {
            float b = lane < kSWarps ? sh.best_s[par][st][sd][lane] : -INFINITY;
            int bc = lane < kSWarps ? sh.best_c[par][st][sd][lane] : INT_MAX;
            warp_best(b, bc);
            if (lane == 0) p.tb[t * p.n_seeds + sd] = TileSeed{b, bc};
        }
    }
    const int ac = warp_min_nonneg(lane < kSWarps ? sh.best_a[par][st][lane] : INT_MAX);
    if (lane == 0) {
        p.te[t] = TileEnd{topk ? sh.tile_nk[par][st] : 0, ac};
        sh.tile_nk[par][st] = 0;
    }
}

template <bool MULTI>
__global__ void __launch_bounds__(kSThreads, DRS_P2_MINB) split_pass2(const __grid_constant__ SplitParams p) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    extern __shared__ __align__(128) unsigned char smem[];
    float4* stages = reinterpret_cast<float4*>(smem);
    __shared__ Pipe pp;
    __shared__ __align__(16) unsigned char recs[kStages][kRowEntryMax];
    __shared__ P2Shared<MULTI> sh;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const bool stats = p.stats != 0;
    const bool probs = stats && p.probs_dtype != 0;
    const bool tma = p.vec != 0;
    const TileRange tiles = launch_tiles(p, p.tiles_per_row);
    if (tid < 2 * kStages) sh.tile_nk[tid / kStages][tid % kStages] = 0;
    pipe_start<kTileCols>(p, pp, p.list1, tiles, p.tiles_per_row, stages, &recs[0][0], kRowEntryMax, p.rr,
               static_cast<uint32_t>(p.rec_bytes), tma);
    for (int n = 0;; ++n) {
        const int st = n % kStages;
        const int par = (n / kStages) & 1;
        float4* stage = stages + st * kStageF4;
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&pp.full[st], static_cast<uint32_t>(par)))) {
            if (lane == 0) {
                pp.abort = 1;
                raise_device_error(p.err, 1);
            }
            break;
        }
        const int row = pp.row[n % kMap];
        if (row < 0) break;
        const int64_t t = tiles.t_begin + static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(n) * gridDim.x;
        const int col0 = pp.col[n % kMap] * kTileCols;
        const int ncols = min(p.vocab - col0, kTileCols);
        const bool topk = p2_warp<MULTI>(p, sh, stage, &recs[st][0], row, pp.lrow[n % kMap], t, col0, ncols, st,
                                         par, tid, lane, warp, stats, probs, tma);
        if (!release_stage(&pp.count[st], lane)) continue;

        // the last warp out: the tile's records (the row entry in the stage
        // is read first), then refill the stage
        p2_combine<MULTI>(p, sh, t, st, par, stats, topk, lane);
        __syncwarp();
        pipe_advance<kTileCols>(p, pp, n, p.list1, tiles, p.tiles_per_row, stage, &recs[st][0], p.rr,
                     static_cast<uint32_t>(p.rec_bytes), tma, lane);
    }
    asm volatile("griddepcontrol.launch_dependents;");
    pipe_end(pp);
}

// ============================================================== finish

// KU: tile counts per lane (rows of up to 60 tiles, and the longest rows)
template <int KU>
__global__ void __launch_bounds__(kRowWarps * 32) split_finish(const __grid_constant__ SplitParams p) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __shared__ uint64_t keys[kRowWarps][kRowKeys];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int64_t li = static_cast<int64_t>(blockIdx.x) * kRowWarps + warp;
    if (li >= p.hard[kCount1]) return;
    const int64_t row = p.list1[li];
    const int G = p.tiles_per_row;
    const unsigned char* entry = p.rr + row * p.rec_bytes;
    const RowRecord rec = *reinterpret_cast<const RowRecord*>(entry);
    const SeedRec* seeds = reinterpret_cast<const SeedRec*>(entry + sizeof(RowRecord));
    const TileEnd* te = p.te + li * G;
    if (p.stats) {
        // argmax: the lowest column holding the raw max, or a lower one
        // whose exact quotient ties it; per seed the sample: the best of the
        // tiles' race winners and B (greedy rows: the argmax)
        int a = rec.arg;
        for (int c = lane; c < G; c += 32) a = min(a, te[c].acol);
        a = warp_min_nonneg(a);
        if (lane == 0) p.argmax[row] = a;
        for (int sd = 0; sd < p.n_seeds; ++sd) {
            float b = seeds[sd].B;
            int bc = seeds[sd].bcol;
            for (int c = lane; c < G; c += 32) {
                const TileSeed e = p.tb[(li * G + c) * p.n_seeds + sd];
                if (beats(e.b, e.col, b, bc)) {
                    b = e.b;
                    bc = e.col;
                }
            }
            warp_best(b, bc);
            if (lane == 0)
                p.sample[sd * p.rows + row] = (rec.flags & kFNoisy) && b != -INFINITY ? bc : a;
        }
    }
    if (!(rec.flags & kFTopk)) return;
    // the row's candidates: counts, then the keys gathered in tile order
    constexpr int kU = KU;
    int n[kU], off[kU];
    bool over_l = false;
#pragma unroll
    for (int u = 0; u < kU; ++u) {
        const int c = lane + 32 * u;
        // (clamped: records of a call whose bounded waits ran out may hold
        // anything; a count past kTileKeys sends the row to the exact kernel)
        n[u] = c < G ? min(max(te[c].nk, 0), kTileKeys + 1) : 0;
        over_l |= n[u] > kTileKeys;
    }
    const bool over = __any_sync(0xffffffffu, over_l);
    int total = 0;
#pragma unroll
    for (int u = 0; u < kU; ++u) {
        int incl = n[u];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += y;
        }
        off[u] = total + incl - n[u];
        total += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (over || total > kRowKeys || total < p.k) {
        if (lane == 0) {
            const int idx = atomicAdd(p.hard, 1);
            p.hard[kHardOffset + idx] = static_cast<int32_t>(row);
        }
        return;
    }
    uint64_t* kw = keys[warp];
    for (int c = 0; c < G; ++c) {
        int nsel = 0, osel = 0;
#pragma unroll
        for (int u = 0; u < kU; ++u)
            if ((c >> 5) == u) {
                nsel = n[u];
                osel = off[u];
            }
        const int nc = __shfl_sync(0xffffffffu, nsel, c & 31);
        const int oc = __shfl_sync(0xffffffffu, osel, c & 31);
        const uint64_t* src = p.keys + (li * G + c) * kTileKeys;
        if (lane < nc) kw[oc + lane] = src[lane];
    }
    __syncwarp();
    const int K = p.k;
    for (int a = lane; a < total; a += 32) {
        const uint64_t key = kw[a];
        int rank = 0;
        for (int o = 0; o < total; ++o) rank += kw[o] > key;
        if (rank < K) {
            p.out_ids[row * K + rank] = key_col(key);
            p.out_lp[row * K + rank] = rec.M == -INFINITY ? NAN : (key_value(key) - rec.M) - rec.lns;
        }
    }
}

// ============================================================== gather

// Top-k calls read each row once. Pass 1 records every warp's raw max; the
// merge takes the row's threshold from them (the k-th largest, lowered by
// Te ulp). A logit at or above the threshold lies in a warp whose max
// reaches it, so this kernel reads back only those warps' columns (the
// "hot" warps: about k of a row's 344 on the step recipe, a few percent of
// its bytes), keys the logits at or above the threshold by (exact value,
// lower column), ranks them by counting and writes the row's top k. A row
// with more hot warps or candidates than fit goes on the hard-row list.
constexpr int kHotCap = 256;  // hot warps a row may have

__global__ void __launch_bounds__(256) split_gather(const __grid_constant__ SplitParams p) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __shared__ uint16_t hot[kHotCap];
    __shared__ uint64_t keys[kRowKeys];
    __shared__ int nhot, nkeys;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int64_t li = blockIdx.x;
    if (li >= p.hard[kCount1]) return;
    const int64_t row = p.list1[li];
    const RowRecord rec = *reinterpret_cast<const RowRecord*>(p.rr + row * p.rec_bytes);
    if (!(rec.flags & kFTopk)) return;  // no threshold: the exact kernel takes the row
    const float thr = rec.thr;
    const uint32_t thr_key = ord32(thr);
    const int G1 = p.tiles1;
    const TileStats* tr = p.ts + li * G1;
    if (tid == 0) {
        nhot = 0;
        nkeys = 0;
    }
    __syncthreads();
    for (int j = tid; j < G1 * kSWarps; j += 256) {
        const uint32_t wm = tr[j / kSWarps].wmax[j % kSWarps];  // 0: a warp without columns
        if (wm != 0u && wm >= thr_key) {
            const int at = atomicAdd(&nhot, 1);
            if (at < kHotCap) hot[at] = static_cast<uint16_t>(j);
        }
    }
    __syncthreads();
    const int nh = nhot;
    if (nh <= kHotCap) {
        const int64_t lrow = p.map_row ? p.map_row[row] : row;
        const float* xr = p.logits + lrow * p.row_stride;
        const ScaledQuotient sq{rec.qt, rec.qy, rec.qmode};
        for (int h = warp; h < nh; h += kSWarps) {
            const int j = hot[h];
            const int w = j % kSWarps;
            const int col0 = (j / kSWarps) * kP1Cols;
#pragma unroll
            for (int i = 0; i < kP1Vec4; ++i) {
                // slot i of the warp's lane: float4 i * kSThreads + 32 w + lane of the tile
                const int c = col0 + 4 * (i * kSThreads + 32 * w + lane);
                if (c >= p.vocab) continue;
                float4 x4;
                if (p.vec && c + 4 <= p.vocab) {
                    x4 = __ldcs(reinterpret_cast<const float4*>(xr + c));
                } else {
                    x4 = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
                    for (int q = 0; q < 4 && c + q < p.vocab; ++q) set_comp(x4, q, __ldcs(xr + c + q));
                }
                if (max4f(x4) >= thr) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float x = comp(x4, q);
                        if (x >= thr) {
                            const int at = atomicAdd(&nkeys, 1);
                            if (at < kRowKeys) keys[at] = topk_key(sq.exact(x), c + q);
                        }
                    }
                }
            }
        }
    }
    __syncthreads();
    const int n = nkeys;
    if (nh > kHotCap || n > kRowKeys || n < p.k) {
        if (tid == 0) {
            const int idx = atomicAdd(p.hard, 1);
            p.hard[kHardOffset + idx] = static_cast<int32_t>(row);
        }
        return;
    }
    const int K = p.k;
    for (int a = tid; a < n; a += 256) {
        const uint64_t key = keys[a];
        int rank = 0;
        for (int o = 0; o < n; ++o) rank += keys[o] > key;
        if (rank < K) {
            p.out_ids[row * K + rank] = key_col(key);
            p.out_lp[row * K + rank] = rec.M == -INFINITY ? NAN : (key_value(key) - rec.M) - rec.lns;
        }
    }
}

// ================================================================ host

size_t round_up(size_t n, size_t a) { return (n + a - 1) / a * a; }

struct SplitLayout {
    size_t hard, list1, rt, ts, rr, te, tb, keys, total;
};

size_t row_entry_bytes(int32_t n_seeds) {
    return sizeof(RowRecord) + static_cast<size_t>(n_seeds) * sizeof(SeedRec);
}

SplitLayout split_layout(int64_t rows, int64_t vocab, int32_t k, int32_t n_seeds) {
    const size_t R = static_cast<size_t>(rows);
    const size_t G = static_cast<size_t>((vocab + kTileCols - 1) / kTileCols);  // pass-2 tiles
    const size_t G1 = static_cast<size_t>((vocab + kP1Cols - 1) / kP1Cols);      // pass-1 tiles
    SplitLayout l{};
    size_t at = 0;
    l.hard = at;
    at += round_up(4 * (kHardOffset + R), kWorkspaceAlign);
    l.list1 = at;
    at += round_up(4 * R, kWorkspaceAlign);
    l.rt = at;
    at += round_up(sizeof(RowTemp) * R, kWorkspaceAlign);
    l.ts = at;
    at += round_up(sizeof(TileStats) * R * G1, kWorkspaceAlign);
    l.rr = at;
    at += round_up(row_entry_bytes(n_seeds) * R, kWorkspaceAlign);
    l.te = at;
    at += round_up(sizeof(TileEnd) * R * G, kWorkspaceAlign);
    l.tb = at;
    at += round_up(sizeof(TileSeed) * R * G * static_cast<size_t>(n_seeds), kWorkspaceAlign);
    l.keys = at;
    if (k > 0) at += round_up(8 * R * G * kTileKeys, kWorkspaceAlign);
    l.total = at;
    return l;
}

template <typename Kernel>
int resident_grid(Kernel kernel, int threads, size_t smem) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess)
        return 0;
    return per_sm * sm_count();
}

}  // namespace

size_t split_workspace_bytes(int64_t rows, int64_t vocab, int32_t k, int32_t n_seeds) {
    return split_layout(rows, vocab, k, n_seeds).total;
}

SplitPrepTargets split_prep_targets(void* workspace, int64_t rows, int64_t vocab, int32_t k, int32_t n_seeds) {
    const SplitLayout l = split_layout(rows, vocab, k, n_seeds);
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    return SplitPrepTargets{reinterpret_cast<int32_t*>(ws + l.hard), reinterpret_cast<int32_t*>(ws + l.list1),
                            ws + l.rt};
}

int32_t split_max_seeds() { return kMaxSeeds; }

int32_t split_max_k() { return kSplitMaxK; }

bool rs::row_split_plan(int64_t rows, int64_t vocab, int32_t k, int32_t n_seeds, bool aligned16,
                        int probs_dtype, bool stats, RowSplitPlan* out) {
    RowSplitPlan pl{};
    if (!stats) return false;  // top-k calls: pass 1 and the gather (one read)
    if (!cluster_plan(rows, vocab, k, n_seeds, aligned16, &pl.shape, &pl.cluster_size)) return false;
    pl.clusters = cluster_active(probs_dtype, pl.cluster_size);
    if (pl.clusters < 1) return false;
    pl.free_sms = sm_count() - pl.clusters * pl.cluster_size;
    // rows per SM and time: the two passes about 10/13 of the cluster
    // kernel's (the best of a sweep of this weight on the step workload), so
    // the tail gets that share of the free SMs' weight; the head is the rest
    // of the list, whatever its length on the device
    pl.head_num = 1;
    pl.head_den = 1;
    pl.tail = 0;
    if (pl.free_sms >= 8 && rows >= 8 * static_cast<int64_t>(pl.clusters)) {
        pl.head_num = 13 * pl.clusters * pl.cluster_size;
        pl.head_den = 10 * pl.free_sms + pl.head_num;
        pl.tail = rows - rows * pl.head_num / pl.head_den;
    }
    *out = pl;
    return true;
}

bool split_plan_query(int64_t rows, int64_t vocab, int32_t k, int32_t n_seeds, bool aligned16, int probs_dtype,
                      bool stats, int64_t* head, int32_t* cluster_size, int32_t* clusters, int32_t* free_sms) {
    RowSplitPlan pl{};
    if (two_pass_forced() || !rs::row_split_plan(rows, vocab, k, n_seeds, aligned16, probs_dtype, stats, &pl))
        return false;
    *head = rows - pl.tail;
    *cluster_size = pl.cluster_size;
    *clusters = pl.clusters;
    *free_sms = pl.free_sms;
    return true;
}

drs_status split_rows(const RowCall& c, void* workspace, cudaStream_t stream) {
    if (c.rows <= 0) return DRS_OK;
    if (c.k > kSplitMaxK || c.vocab > DRS_MAX_VOCAB) return DRS_ERR_UNSUPPORTED;
    const int32_t n_seeds = c.seeds ? c.n_seeds : 1;
    if (n_seeds < 1 || n_seeds > kMaxSeeds) return DRS_ERR_UNSUPPORTED;
    const int G = static_cast<int>((c.vocab + kTileCols - 1) / kTileCols);  // pass-2 tiles per row
    const int G1 = static_cast<int>((c.vocab + kP1Cols - 1) / kP1Cols);     // pass-1 tiles per row
    // tile indices of a pass are 32-bit, list lengths int
    if (c.rows > INT_MAX / G1) return DRS_ERR_UNSUPPORTED;
    const SplitLayout l = split_layout(c.rows, c.vocab, c.k, n_seeds);
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    SplitParams p{};
    p.logits = c.logits;
    p.row_stride = c.row_stride;
    p.rows = c.rows;
    p.row0 = c.row0;
    p.canvas_len = c.canvas_len;
    p.temps = c.temps;
    p.keep = c.keep;
    p.argmax = c.argmax;
    p.sample = c.sample;
    p.entropy = c.entropy;
    p.probs = c.probs;
    p.probs_row_stride = c.probs_row_stride;
    p.out_ids = c.out_ids;
    p.out_lp = c.out_lp;
    p.hard = reinterpret_cast<int32_t*>(ws + l.hard);
    p.list1 = reinterpret_cast<int32_t*>(ws + l.list1);
    p.rt = reinterpret_cast<RowTemp*>(ws + l.rt);
    p.ts = reinterpret_cast<TileStats*>(ws + l.ts);
    p.rr = ws + l.rr;
    p.te = reinterpret_cast<TileEnd*>(ws + l.te);
    p.tb = reinterpret_cast<TileSeed*>(ws + l.tb);
    p.keys = reinterpret_cast<uint64_t*>(ws + l.keys);
    p.map_row = c.map_row;
    p.map_temp = c.map_temp;
    p.map_count = c.map_count;
    p.out_m = c.out_m;
    p.out_logs = c.out_logs;
    p.err = device_error_flag();
    if (!p.err) return DRS_ERR_CUDA;
    for (int sd = 0; sd < n_seeds; ++sd)
        p.rk[sd] = PhiloxRoundKeys::of(c.seeds ? c.seeds[sd] : c.seed);
    p.n_seeds = n_seeds;
    p.rec_bytes = static_cast<int>(row_entry_bytes(n_seeds));
    p.tiles_per_row = G;
    p.tiles1 = G1;
    p.vocab = static_cast<int>(c.vocab);
    p.vec = aligned(c.logits, 16) && (c.row_stride % 4 == 0);
    p.probs_dtype = static_cast<int>(c.probs_dtype);
    p.probs_vec = c.probs && aligned(c.probs, 8) && (c.probs_row_stride % 4 == 0);
    p.index32 = (c.row0 + c.rows <= static_cast<int64_t>(UINT32_MAX)) &&
                (c.canvas_len <= static_cast<int64_t>(UINT32_MAX));
    p.stats = c.stats ? 1 : 0;
    p.k = c.k;
    p.li_part = 0;
    p.li_num = 1;
    p.li_den = 1;
    p.fault = take_injected_fault();
    const size_t smem = kStages * kStageBytes;                       // pass 2
    const size_t smem1 = static_cast<size_t>(kStages) * kP1Cols * 4;  // pass 1
    const int64_t gp = (c.rows + 255) / 256;
    const int64_t gr = (c.rows + kRowWarps - 1) / kRowWarps;
    if (gr > INT_MAX) return DRS_ERR_UNSUPPORTED;
    // with kernel timing on, an event before each kernel and after the last
    const int slot = kernel_timer_slot();
    auto mark = [&](int i) {
        return slot < 0 || cudaEventRecord(kernel_timer_event(slot, i), stream) == cudaSuccess;
    };
    auto pass2 = n_seeds > 1 ? split_pass2<true> : split_pass2<false>;
    if (cudaFuncSetAttribute(split_pass1, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem1)) != cudaSuccess ||
        cudaFuncSetAttribute(pass2, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return DRS_ERR_CUDA;
    const int g1 = resident_grid(split_pass1, kSThreads, smem1);
    const int g2 = resident_grid(pass2, kSThreads, smem);
    if (g1 < 1 || g2 < 1) return DRS_ERR_CUDA;
    if (!mark(0)) return DRS_ERR_CUDA;
    if (!c.prepared) split_prep<<<static_cast<int>(gp), 256, 0, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess || !mark(1)) return DRS_ERR_CUDA;
    // pass 1, merge, pass 2 and finish may launch while their predecessor
    // drains (each waits for it before its first access)
    auto pdl = [&](auto kernel, int grid, int block, size_t dsmem) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(block);
        cfg.dynamicSmemBytes = dsmem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kernel, p) == cudaSuccess;
    };
    // One read per row where the cluster kernel takes the call. Its clusters
    // of up to 16 CTAs (one per SM) fit only the GPU's larger SM groups; on a
    // large enough call the SMs they leave free run the two passes over the
    // tail of the row list at the same time, on a second stream (the two
    // parts fill one workspace, one finish kernel reduces both). Else the two
    // passes alone.
    if (!c.stats && c.k > 0) {
        // top-k calls read each row once: pass 1, the merge's threshold,
        // then only the columns of the warps whose max reaches it (the
        // finish's event slot times the gather)
        const bool short_m = G1 * kSWarps <= 32 * kOrdSmall;
        if (!pdl(split_pass1, g1, kSThreads, smem1) || !mark(2)) return DRS_ERR_CUDA;
        const bool ok = short_m ? pdl(split_merge<kOrdSmall, 1>, static_cast<int>(gr), kRowWarps * 32, 0)
                                : pdl(split_merge<kOrdWide, kWideMergeWarps>, static_cast<int>(c.rows),
                                      kRowWarps * 32, 0);
        if (!ok || !mark(3) || !mark(4) || !mark(5)) return DRS_ERR_CUDA;
        if (c.rows > INT_MAX || !pdl(split_gather, static_cast<int>(c.rows), 256, 0) || !mark(6))
            return DRS_ERR_CUDA;
        return DRS_OK;
    }
    RowSplitPlan plan{};
    if (!two_pass_forced() &&
        rs::row_split_plan(c.rows, c.vocab, c.k, n_seeds, p.vec != 0, p.probs_dtype, c.stats, &plan)) {
        const ClusterShape cshape = plan.shape;
        const int csize = plan.cluster_size;
        const int free_sms = plan.free_sms;
        int64_t tail = plan.tail;
        cudaStream_t side = nullptr;
        cudaEvent_t fork = nullptr, join = nullptr;
        if (tail > 0 && !side_stream(&side, &fork, &join)) tail = 0;
        const int64_t head = c.rows - tail;
        p.tiles_per_row = G;
        if (!mark(2) || !mark(3) || !mark(4)) return DRS_ERR_CUDA;
        if (tail > 0) {
            // the two passes over the tail of the list beside the cluster
            // kernel, their persistent grids sized for the free SMs
            if (cudaEventRecord(fork, stream) != cudaSuccess || cudaStreamWaitEvent(side, fork, 0) != cudaSuccess)
                return DRS_ERR_CUDA;
            SplitParams q = p;
            q.li_part = 2;
            q.li_num = plan.head_num;
            q.li_den = plan.head_den;
            q.tiles_per_row = G;
            auto pdl_side = [&](auto kernel, int grid, int block, size_t dsmem) {
                cudaLaunchConfig_t cfg = {};
                cfg.gridDim = dim3(grid);
                cfg.blockDim = dim3(block);
                cfg.dynamicSmemBytes = dsmem;
                cfg.stream = side;
                cudaLaunchAttribute attr[1];
                attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
                attr[0].val.programmaticStreamSerializationAllowed = 1;
                cfg.attrs = attr;
                cfg.numAttrs = 1;
                return cudaLaunchKernelEx(&cfg, kernel, q) == cudaSuccess;
            };
            const int gq1 = std::min(g1, 3 * free_sms);
            const int gq2 = std::min(g2, 3 * free_sms);
            const int64_t gt = (tail + kRowWarps - 1) / kRowWarps;
            const bool short_m = G1 * kSWarps <= 32 * kOrdSmall;
            if (!pdl_side(split_pass1, gq1, kSThreads, smem1) ||
                !(short_m ? pdl_side(split_merge<kOrdSmall, 1>, static_cast<int>(gt), kRowWarps * 32, 0)
                          : pdl_side(split_merge<kOrdWide, kWideMergeWarps>, static_cast<int>(tail), kRowWarps * 32,
                                     0)) ||
                !pdl_side(pass2, gq2, kSThreads, smem) || cudaEventRecord(join, side) != cudaSuccess)
                return DRS_ERR_CUDA;
        }
        SplitParams pc = p;
        if (tail > 0) {
            pc.li_part = 1;
            pc.li_num = plan.head_num;
            pc.li_den = plan.head_den;
        }
        if (cluster_launch(pc, cshape, csize, head, stream) != DRS_OK || !mark(5)) return DRS_ERR_CUDA;
        if (tail > 0 && cudaStreamWaitEvent(stream, join, 0) != cudaSuccess) return DRS_ERR_CUDA;
        auto finish = G <= 32 * kTilesSmall ? split_finish<kTilesSmall> : split_finish<kTilesLarge>;
        if (!pdl(finish, static_cast<int>(gr), kRowWarps * 32, 0) || !mark(6)) return DRS_ERR_CUDA;
        return DRS_OK;
    }
    if (!pdl(split_pass1, g1, kSThreads, smem1) || !mark(2)) return DRS_ERR_CUDA;
    const bool short_merge = G1 * kSWarps <= 32 * kOrdSmall;
    const bool ok3 = short_merge ? pdl(split_merge<kOrdSmall, 1>, static_cast<int>(gr), kRowWarps * 32, 0)
                                 : pdl(split_merge<kOrdWide, kWideMergeWarps>, static_cast<int>(c.rows),
                                       kRowWarps * 32, 0);
    if (!ok3 || !mark(3)) return DRS_ERR_CUDA;
    if (!pdl(pass2, g2, kSThreads, smem) || !mark(4) || !mark(5)) return DRS_ERR_CUDA;
    auto finish = G <= 32 * kTilesSmall ? split_finish<kTilesSmall> : split_finish<kTilesLarge>;
    if (!pdl(finish, static_cast<int>(gr), kRowWarps * 32, 0) || !mark(6)) return DRS_ERR_CUDA;
    return DRS_OK;
}

}  // namespace drs
