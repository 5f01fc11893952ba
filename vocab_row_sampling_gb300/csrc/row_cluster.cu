// row_cluster.cu -- the row statistics with ONE read of the logits (page
// "vllm.model_executor.models.diffusion_gemma_sampler": the module docstring's
// single read with an online max and sum, the noise drawn inline and one write
// of the probabilities; sample_row_stats_reference for what is computed).
//
// A row is split over the C CTAs of a thread-block cluster (one CTA per SM),
// each owning a contiguous chunk of at most 16384 columns (64 KiB) that stays
// in its shared memory from the bulk copy (TMA) that brings it in until the
// probabilities have been written from it. A CTA holds three rows at once in
// a ring of three chunk buffers and runs four kinds of warps:
//   16 compute warps: for row t, phase A -- per warp, the raw max and its
//            lowest column, S = sum e^(s - m) and W = sum e^(s - m)(s - m)
//            (raw-domain exponentials while |m| < 256, exact quotients
//            beyond) -- then, for row t - 1 whose merged statistics are
//            ready, phase B -- the probabilities, the argmax ties, the
//            pruned Gumbel race against B, the top-k candidates;
//   the merge warp: combines the compute warps' phase-A results into the
//            CTA's part (m, S, W, raw max and column, the CTA's largest group
//            maxima, the best Gumbel-max score of its warps' argmax
//            elements), pushes it into every CTA of the cluster (st.async
//            into distributed shared memory, completing on each receiver's
//            mbarrier) and merges the C parts of the row once they have
//            landed (the row's M, S, W, argmax column and B);
//   the noise warp: the Gumbel-max scores of the warps' argmax elements
//            for the part, then the row's top-k threshold from the parts;
//   the feed warp: the ring of row entries, the bulk copies into the
//            buffers, and after phase B the CTA's race winner, argmax tie
//            and candidate count, before it starts the copy of row t + 3
//            into the freed buffer.
// The compute warps never wait for the exchange of their current row: while
// it runs they work on the previous one. The CTA's results go to the same
// per-tile records the two-pass kernels write (a CTA is one tile of its row),
// and the finish kernel of row_split.cu reduces them.
//
// HBM traffic: every logit read once, every probability written once.
#include "row_common.cuh"

namespace drs {
namespace rs {
namespace {

constexpr int kCompWarps = 16;                      // compute warps per CTA
constexpr int kCompThreads = kCompWarps * 32;       // 512
// The control warps come first: warps of lower index win the scheduler's
// choice among ready warps, and the control warps' short serial chains pace
// every row.
constexpr int kMergeWarp = 0;                       // the CTA's part and the row merge
constexpr int kFeedWarp = 1;                        // row ring, copies, per-tile records
constexpr int kNoiseWarp = 2;                       // Gumbel candidates, top-k threshold
constexpr int kCtlWarps = 3;
constexpr int kCThreads = kCompThreads + 32 * kCtlWarps;  // compute warps 3 .. 18
constexpr int kCRing = 128;                         // rows of the ring (filled 32 at a time)
constexpr int kCSlots = 8;                          // float4 per compute thread and row
constexpr int kCChunkF4 = kCompThreads * kCSlots;   // 4096 float4 per chunk
constexpr int kCChunkMax = 4 * kCChunkF4;           // 16384 columns per CTA
constexpr int kCMaxCluster = 16;
constexpr int kCBufs = 3;                           // rows held per CTA
constexpr int kCGroups = kCompWarps;                // group maxima per CTA (a warp's 1024 columns)
// Part slots, by row iteration t % kCPartSlots. Three make reuse safe by
// causality: a CTA pushes row t + 3 only after all C parts of row t + 1 have
// reached it, and a CTA pushes its part of row t + 1 only after it has
// finished reading the parts of row t.
constexpr int kCPartSlots = 3;

// A CTA's phase-A part of a row (96 bytes), pushed to every CTA of the
// cluster.
struct alignas(16) CPart {
    float m;      // max exact quotient of the CTA's columns (-inf: none)
    float s;      // sum e^(s - m)
    float w;      // sum e^(s - m) (s - m)
    float xmax;   // raw max
    int arg;      // lowest column holding it (the CTA's first column if none)
    float bs;     // best Gumbel-max score of the warps' argmax elements
    int bc;       // its column
    int ng;       // group maxima below
    uint32_t gm[kCGroups];  // the CTA's largest group maxima (order keys), descending; 0 past ng
};
static_assert(sizeof(CPart) == 96, "CTA part");
// 16-byte words of a part that a row pushes: the statistics (32 bytes), and
// for a top-k row the first top_m group maxima.
__device__ __forceinline__ uint32_t part_words(bool topk, int top_m) {
    return 2u + (topk ? static_cast<uint32_t>(top_m + 3) / 4u : 0u);
}

// The merged row as phase B uses it.
struct alignas(16) CRow {
    float M, log2s, ls, c2, thr, cthr, B, cB, xB;
    float qt, qy;
    int qmode, flags, bcol, pad0, pad1;
};

// A row of the cluster's list as every warp of the CTA reads it (32 bytes):
// filled by the feed warp, 32 rows at a time, ahead of the row's copy.
struct alignas(16) RowSlot {
    int row;      // the call's row (list entry)
    int lrow;     // its logits row (differs under a row map)
    float temp;   // T (not clamped)
    int kept;     // the row's slot is converged (its top-k is wanted)
    float qt, qy;
    int qmode;
    int pad;
};

// A compute warp's phase-B result for a row.
struct alignas(16) WarpRes {
    float b;   // best race score
    int c;     // its column
    int a;     // lowest column below the raw max whose exact quotient is M
    int pad;
};

struct ClusterSmem {
    uint64_t full[kCBufs];   // a buffer's row landed (TMA)
    uint64_t adone[2];       // the compute warps' phase A of a row (by row parity)
    uint64_t recrdy[2];      // the merged row is ready for phase B
    uint64_t bdone[2];       // the compute warps' phase B of a row
    uint64_t part_full[kCPartSlots];  // the C parts of a row landed
    uint64_t cand_done[2];   // the noise warp scored the CTA's Gumbel candidates
    uint64_t thr_done[2];    // the noise warp set the row's top-k threshold
    int abort;
    int tile_nk[2];          // top-k candidates of the CTA, by row parity
    int issued[kCBufs];      // row iteration last copied into each buffer (-1: none)
    RowSlot ring[kCRing];    // row iteration t at t % kCRing
    CPart part[kCPartSlots][kCMaxCluster];
    CPart mine;
    WarpPart wparts[2][kCompWarps];
    WarpRes wres[2][kCompWarps];
    CRow row[2];
    float cand_s[2];         // best Gumbel-max score of the CTA's candidates
    int cand_c[2];           // its column
    uint16_t race_at[kCompWarps][kCSlots * 32];
};

// ------------------------------------------------------ cluster PTX

__device__ __forceinline__ uint32_t cta_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cta_count() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_index() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_total() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster arrives; returns once all have
// (release / acquire at cluster scope). Used once, after the mbarriers are
// initialised: all CTAs of a cluster are resident together, so it completes.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The shared::cluster address of the same shared-memory location in CTA
// `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t smem_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
    return r;
}

// 16 bytes into another CTA's shared memory, counted as transaction bytes on
// that CTA's mbarrier.
__device__ __forceinline__ void push16(uint32_t remote_addr, const uint4& v, uint32_t remote_bar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
            remote_addr),
        "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(remote_bar)
        : "memory");
}

__device__ __forceinline__ bool try_wait_cluster(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return done != 0;
}

// Wait for the phase of `bar` with the given parity (acquire at CTA scope,
// or at cluster scope for barriers completed by other CTAs' pushes). Gives
// up -- false -- after kWaitLimitNs, or as soon as another warp of the CTA
// has given up (abort set): a wait never outlives a failed one for long.
template <bool CLUSTER>
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, const volatile int* abort) {
    if (CLUSTER ? try_wait_cluster(bar, parity, 2000u) : mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (CLUSTER ? try_wait_cluster(bar, parity, 1000000u) : mbar_try_wait_suspend(bar, parity, 1000000u))
            return true;
        if (*abort) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// The noise warp waits for the same phase of part_full as the merge warp (a
// phase can be waited on by any number of threads; the merge warp re-arms
// the barrier only after the noise warp has passed it for this row).
__device__ __forceinline__ bool try_wait_parts(ClusterSmem& sh, int ps, uint32_t ppar) {
    return wait_phase<true>(&sh.part_full[ps], ppar, &sh.abort);
}

__device__ __forceinline__ void give_up(ClusterSmem& sh, int* err) {
    sh.abort = 1;
    __threadfence_block();
    raise_device_error(err, 1);
}

// ------------------------------------------------------ rows

// The list entries of this cluster are li0, li0 + ncl, ...; entry t of them
// is row iteration t. The feed warp fills ring entries [t0, t0 + 32) (one
// per lane: three dependent loads per row, in parallel over the lanes).
__device__ __forceinline__ void fill_ring(const SplitParams& p, ClusterSmem& sh, int li0, int ncl, int T, int t0,
                                          int lane) {
    const int t = t0 + lane;
    if (t >= T) return;
    RowSlot rs;
    rs.row = p.list1[li0 + t * ncl];
    rs.lrow = p.map_row ? p.map_row[rs.row] : rs.row;
    const RowTemp rt = p.rt[rs.row];
    rs.temp = rt.temp;
    rs.qt = rt.qt;
    rs.qy = rt.qy;
    rs.qmode = rt.qmode;
    rs.kept = p.map_row || p.keep == nullptr ||
              p.keep[slot_of(p, static_cast<uint64_t>(p.row0 + rs.row))] != 0;
    rs.pad = 0;
    sh.ring[t % kCRing] = rs;
}

// Copy the CTA's chunk of row iteration it (its ring entry filled) into
// buffer b.
__device__ __forceinline__ void issue_row(const SplitParams& p, ClusterSmem& sh, float4* buf, int b, int it,
                                          int c0, int ncols) {
    sh.issued[b] = it;
    if (p.fault && it == 0 && blockIdx.x == 0) {
        // the test hook: this row never lands, the waits on it run out
        sh.issued[b] = -1;
        return;
    }
    const int64_t lrow = sh.ring[it % kCRing].lrow;
    const uint32_t bytes = static_cast<uint32_t>(ncols) * 4u;
    mbar_arrive_expect_tx(&sh.full[b], bytes);
    tma_load_1d(buf + b * kCChunkF4, p.logits + lrow * p.row_stride + c0, bytes, &sh.full[b]);
}

// ------------------------------------------------------ phase A

// S = sum 2^t and W = ln2 * sum 2^t t, t = x * ls - cref, over a thread's 32
// logits, two at a time; with CLAMP, t is kept finite (a -inf logit gives
// e = 0 and e * t = 0 instead of NaN).
template <bool CLAMP>
__device__ __forceinline__ void sums2(const float4 (&v)[kCSlots], float ls, float cref, float& sw, float& ww) {
    const float2 l2 = make_float2(ls, ls), n2 = make_float2(-cref, -cref);
    float2 sa = make_float2(0.0f, 0.0f), sb = sa, wa = sa, wb = sa;
#pragma unroll
    for (int i = 0; i < kCSlots; ++i) {
        float2 t01 = __ffma2_rn(make_float2(v[i].x, v[i].y), l2, n2);
        float2 t23 = __ffma2_rn(make_float2(v[i].z, v[i].w), l2, n2);
        if (CLAMP) {
            t01 = make_float2(fmaxf(t01.x, -FLT_MAX), fmaxf(t01.y, -FLT_MAX));
            t23 = make_float2(fmaxf(t23.x, -FLT_MAX), fmaxf(t23.y, -FLT_MAX));
        }
        const float2 e01 = make_float2(ex2_ftz(t01.x), ex2_ftz(t01.y));
        const float2 e23 = make_float2(ex2_ftz(t23.x), ex2_ftz(t23.y));
        sa = __fadd2_rn(sa, e01);
        sb = __fadd2_rn(sb, e23);
        wa = __ffma2_rn(e01, t01, wa);
        wb = __ffma2_rn(e23, t23, wb);
    }
    sw = warp_sum_f((sa.x + sa.y) + (sb.x + sb.y));
    ww = warp_sum_f((wa.x + wa.y) + (wb.x + wb.y)) * kLn2;
}

// The rare cases of phase A, out of line: a warp whose largest scaled value
// may reach 256 (exact quotients, t = (s - M_w) log2(e); logits whose
// exponential is 0 anyway are not divided, and a slot none of the warp's
// lanes needs is skipped), and a raw warp holding -inf logits (t clamped:
// 0 * -inf is NaN). Slot by slot, with the accumulation order of sums2.
__device__ __noinline__ void phase_a_rare(const float4* chunk, int ct, const ScaledQuotient& sq, float mxw,
                                          bool raw, float& sw, float& ww) {
    const float yl = kLog2e * sq.y;
    const float mw = raw ? 0.0f : sq.exact(mxw);
    const FarBelow far(mxw, yl);
    const float2 l2 = raw ? make_float2(yl, yl) : make_float2(kLog2e, kLog2e);
    const float2 n2 = raw ? make_float2(-mxw * yl, -mxw * yl) : make_float2(-0.0f, -0.0f);
    float2 sa = make_float2(0.0f, 0.0f), sb = sa, wa = sa, wb = sa;
#pragma unroll 2
    for (int i = 0; i < kCSlots; ++i) {
        float4 v = chunk[i * kCompThreads + ct];
        if (!raw) {
            const bool f0 = far(v.x), f1 = far(v.y), f2 = far(v.z), f3 = far(v.w);
            if (__any_sync(0xffffffffu, !(f0 && f1 && f2 && f3))) {
                v.x = f0 ? kFarStandIn : sq.exact(v.x) - mw;
                v.y = f1 ? kFarStandIn : sq.exact(v.y) - mw;
                v.z = f2 ? kFarStandIn : sq.exact(v.z) - mw;
                v.w = f3 ? kFarStandIn : sq.exact(v.w) - mw;
            } else {
                v = make_float4(kFarStandIn, kFarStandIn, kFarStandIn, kFarStandIn);
            }
        }
        float2 t01 = __ffma2_rn(make_float2(v.x, v.y), l2, n2);
        float2 t23 = __ffma2_rn(make_float2(v.z, v.w), l2, n2);
        if (raw) {
            t01 = make_float2(fmaxf(t01.x, -FLT_MAX), fmaxf(t01.y, -FLT_MAX));
            t23 = make_float2(fmaxf(t23.x, -FLT_MAX), fmaxf(t23.y, -FLT_MAX));
        }
        const float2 e01 = make_float2(ex2_ftz(t01.x), ex2_ftz(t01.y));
        const float2 e23 = make_float2(ex2_ftz(t23.x), ex2_ftz(t23.y));
        sa = __fadd2_rn(sa, e01);
        sb = __fadd2_rn(sb, e23);
        wa = __ffma2_rn(e01, t01, wa);
        wb = __ffma2_rn(e23, t23, wb);
    }
    sw = warp_sum_f((sa.x + sa.y) + (sb.x + sb.y));
    ww = warp_sum_f((wa.x + wa.y) + (wb.x + wb.y)) * kLn2;
}

// One compute warp's share of a chunk: the raw max M_w of its 1024 columns
// (slot i of compute thread ct is float4 i * 512 + ct) and the lowest column
// holding it, S_w and W_w relative to it (raw domain while |M_w| < 256 for
// sure, else from exact quotients).
__device__ __forceinline__ WarpPart phase_a(const float4* chunk, const ScaledQuotient& sq, int c0, int ct,
                                            bool want_arg) {
    float4 v[kCSlots];
#pragma unroll
    for (int i = 0; i < kCSlots; ++i) v[i] = chunk[i * kCompThreads + ct];
    // the thread's max as a tree (a chain of 16 dependent maxima is slow)
    float m8[kCSlots];
#pragma unroll
    for (int i = 0; i < kCSlots; ++i) m8[i] = max4f(v[i]);
    const float mt = fmaxf(max3(m8[0], m8[1], m8[2]), max3(m8[3], m8[4], max3(m8[5], m8[6], m8[7])));
    const float mxw = warp_max_f(mt);
    int aw = INT_MAX;
    if (want_arg) {
        int arg_t = INT_MAX;
        if (mt == mxw && mxw != -INFINITY) {
            int i0 = 0;
#pragma unroll
            for (int i = kCSlots - 1; i >= 0; --i)
                if (m8[i] == mxw) i0 = i;
            const int f = i0 * kCompThreads + ct;
            const float4 x4 = chunk[f];
            const int q = x4.x == mxw ? 0 : x4.y == mxw ? 1 : x4.z == mxw ? 2 : 3;
            arg_t = c0 + 4 * f + q;
        }
        aw = warp_min_nonneg(arg_t);
    }
    const bool raw = fabsf(mxw * sq.y) < kRawLimit - 1.0f;
    float sw = 0.0f, ww = 0.0f;  // a warp of -inf only: nothing to sum
    if (raw) {
        const float lscale = kLog2e * sq.y;
        sums2<false>(v, lscale, mxw * lscale, sw, ww);
    }
    if ((!raw || isnan(ww)) && mxw != -INFINITY) phase_a_rare(chunk, ct, sq, mxw, raw, sw, ww);
    return WarpPart{0.0f, sw, ww, mxw, aw};
}

// ------------------------------------------------------ control warp

// The CTA's part of row iteration t from the compute warps' parts (lane w <
// 16 holds warp w's), into sh.mine, then pushed into slot t & 1 of every CTA.
__device__ __forceinline__ void make_part(const SplitParams& p, ClusterSmem& sh, const RowSlot& ro, int ncols,
                                          int c0, int top_m, int s, uint32_t rank, uint32_t C, int lane) {
    const ScaledQuotient sq{ro.qt, ro.qy, ro.qmode};
    WarpPart wp = lane < kCompWarps ? sh.wparts[s][lane] : WarpPart{0.0f, 0.0f, 0.0f, -INFINITY, INT_MAX};
    const bool present = lane < kCompWarps && lane * 128 < ncols;
    wp.m = wp.xmax == -INFINITY ? -INFINITY : sq.exact(wp.xmax);
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
    const int a_c = xm == -INFINITY ? c0 : warp_min_nonneg(wp.xmax == xm ? wp.arg : INT_MAX);
    // the CTA's top_m group maxima, descending (absent groups are 0, below
    // every value; -inf is kOrdNegInf)
    uint32_t key = present ? ord32(wp.xmax) : 0u;
    uint32_t mine = 0;
    int ng = 0;
    if (ro.kept && p.k > 0) {
        for (int r = 0; r < top_m; ++r) {
            uint32_t top;
            asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(top) : "r"(key));
            if (top == 0) break;
            if (lane == r) mine = top;
            ++ng;
            const uint32_t holders = __ballot_sync(0xffffffffu, key == top);
            if (lane == __ffs(holders) - 1) key = 0;
        }
    }
    if (lane < kCGroups) sh.mine.gm[lane] = mine;
    if (lane == 0) {
        sh.mine.m = mc;
        sh.mine.s = s_c;
        sh.mine.w = w_c;
        sh.mine.xmax = xm;
        sh.mine.arg = a_c;
        sh.mine.ng = ng;
    }
}

// Push the first nw words of the CTA's part (sh.mine, its candidates filled
// in) into part slot ps of every CTA of the cluster: lane d < C to CTA d.
__device__ __forceinline__ void push_part(ClusterSmem& sh, int ps, uint32_t rank, uint32_t C, uint32_t nw, int lane) {
    __syncwarp();
    if (static_cast<uint32_t>(lane) < C) {
        const uint4* src = reinterpret_cast<const uint4*>(&sh.mine);
        const uint32_t dst = smem_u32(&sh.part[ps][rank]);
        const uint32_t rbar = map_to_rank(smem_u32(&sh.part_full[ps]), static_cast<uint32_t>(lane));
        for (uint32_t q = 0; q < nw; ++q)
            push16(map_to_rank(dst + 16u * q, static_cast<uint32_t>(lane)), src[q], rbar);
    }
}

// The noise warp: the Gumbel-max score of each compute warp's argmax element
// (lane w < 16: warp w's; its exact quotient is M_w), the best of them.
__device__ __forceinline__ void score_candidates(const SplitParams& p, ClusterSmem& sh, const RowSlot& ro,
                                                 bool stats, int s, int lane) {
    float bs = -INFINITY;
    int bc = INT_MAX;
    if (stats && ro.temp > 0.0f) {  // rows that draw no noise need no B
        const ScaledQuotient sq{ro.qt, ro.qy, ro.qmode};
        const WarpPart wp = lane < kCompWarps ? sh.wparts[s][lane] : WarpPart{0.0f, 0.0f, 0.0f, -INFINITY, INT_MAX};
        const bool cand = wp.arg != INT_MAX;
        const int ccol = cand ? wp.arg : 0;
        const uint4 nw =
            noise_group(p.rk[0], static_cast<uint64_t>(p.row0 + ro.row), static_cast<uint32_t>(ccol >> 2));
        const float g = gumbel_of_bits(word_of(nw, ccol & 3));
        bs = cand ? sq.exact(wp.xmax) + g : -INFINITY;
        bc = cand ? wp.arg : INT_MAX;
        warp_best(bs, bc);
    }
    if (lane == 0) {
        sh.cand_s[s] = bs;
        sh.cand_c[s] = bc;
    }
}

// The 64 values (a at position lane, b at position lane + 32) in descending
// order, by a bitonic sorting network across the warp.
__device__ __forceinline__ void sort64_desc(uint32_t& a, uint32_t& b, int lane) {
#pragma unroll
    for (int size = 2; size <= 64; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            if (stride == 32) {
                const uint32_t hi = max(a, b), lo = min(a, b);
                a = hi;
                b = lo;
            } else {
                const uint32_t pa = __shfl_xor_sync(0xffffffffu, a, stride);
                const uint32_t pb = __shfl_xor_sync(0xffffffffu, b, stride);
                const bool lower = (lane & stride) == 0;
                const bool desc_a = (lane & size) == 0;
                const bool desc_b = ((lane + 32) & size) == 0;
                a = (lower == desc_a) ? max(a, pa) : min(a, pa);
                b = (lower == desc_b) ? max(b, pb) : min(b, pb);
            }
        }
    }
}

// The k-th largest of the n values v[0 .. n) (0 = absent; 0 if fewer than
// k are present). n <= 64: a sort; else k rounds of a warp max.
__device__ __forceinline__ uint32_t kth_largest(const CPart* pr, int C, int top_m, int k, int lane) {
    const int n = C * top_m;
    auto at = [&](int idx) -> uint32_t {
        if (idx >= n) return 0u;
        const int c = idx / top_m;
        return pr[c].gm[idx - c * top_m];
    };
    if (n <= 64) {
        uint32_t a = at(lane), b = at(lane + 32);
        sort64_desc(a, b, lane);
        return k <= 32 ? __shfl_sync(0xffffffffu, a, k - 1) : __shfl_sync(0xffffffffu, b, k - 33);
    }
    uint32_t o[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) o[u] = at(lane + 32 * u);
    uint32_t kth = 0;
    for (int rd = 0; rd < k; ++rd) {
        uint32_t lm = 0;
#pragma unroll
        for (int u = 0; u < 8; ++u) lm = max(lm, o[u]);
        uint32_t top;
        asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(top) : "r"(lm));
        kth = top;
        if (top == 0) break;
        const uint32_t holders = __ballot_sync(0xffffffffu, lm == top);
        if (lane == __ffs(holders) - 1) {
            bool done = false;
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (!done && o[u] == top) {
                    o[u] = 0;
                    done = true;
                }
        }
    }
    return kth;
}

// The noise warp: the row's top-k threshold into sh.row[s].thr -- the k-th
// largest of the parts' group maxima (k distinct elements reach it, so the
// row's top k all do), lowered by Te ulp(s): a logit below it whose exact
// quotient equals its quotient is a candidate too (equal values rank by
// column). -inf when there is none (absent, or -inf): the exact kernel
// takes the row.
__device__ __forceinline__ void row_threshold(const SplitParams& p, ClusterSmem& sh, const RowSlot& ro, int top_m,
                                              int s, int ps, uint32_t C, int lane) {
    const uint32_t kth = kth_largest(sh.part[ps], static_cast<int>(C), top_m, p.k, lane);
    float thr = -INFINITY;
    if (kth > kOrdNegInf) {
        const float x = unord32(kth);
        thr = x - fmaxf(fabsf(x) * 0x1p-20f, ro.qt * 0x1p-140f);
    }
    if (lane == 0) sh.row[s].thr = thr;
}

// The row from the C parts in slot s into sh.row[s]. Every CTA computes the
// same; CTA 0 of the cluster also writes the row's record for the finish
// kernel, the entropy, the stash's max and log S, and rows without a
// threshold on the hard list.
__device__ __forceinline__ bool merge_parts(const SplitParams& p, ClusterSmem& sh, const RowSlot& ro, bool stats,
                                            int s, int par, int ps, uint32_t rank, uint32_t C, int lane) {
    const bool topk = ro.kept && p.k > 0;
    const CPart* pr = sh.part[ps];
    float m = -INFINITY, sp = 0.0f, wq = 0.0f, xm = -INFINITY, bs = -INFINITY;
    int arg = INT_MAX, bc = INT_MAX;
    if (lane < static_cast<int>(C)) {
        const CPart& q = pr[lane];
        m = q.m;
        sp = q.s;
        wq = q.w;
        xm = q.xmax;
        arg = q.arg;
        bs = q.bs;
        bc = q.bc;
    }
    const float big_m = warp_max_f(m);
    float s_l = 0.0f, w_l = 0.0f;
    if (m != -INFINITY) {
        const float dm = m - big_m;
        const float f = ex2_approx(dm * kLog2e);
        s_l = f * sp;
        w_l = f * fmaf(dm, sp, wq);
    }
    const float s_tot = warp_sum_f(s_l);
    const float w_tot = warp_sum_f(w_l);
    const float mraw = warp_max_f(xm);
    const int arg_row = warp_min_nonneg(xm == mraw ? arg : INT_MAX);
    warp_best(bs, bc);

    // the top-k threshold, from the noise warp (-inf: none)
    if (topk && !__all_sync(0xffffffffu, wait_phase<false>(&sh.thr_done[s], static_cast<uint32_t>(par), &sh.abort)))
        return false;
    const float thr = topk ? sh.row[s].thr : -INFINITY;
    const bool hard = topk && thr == -INFINITY;
    const bool noisy = stats && ro.temp > 0.0f && big_m != -INFINITY;
    const float ls = kLog2e * ro.qy;
    const float c0 = mraw * ls;
    const float log2s = s_tot > 0.0f ? log2f(s_tot) : 0.0f;
    const bool raw = !(fabsf(big_m) >= kRawLimit);
    const float cB = (c0 + (bs - big_m) * kLog2e) - kRaceSlack;
    if (lane == 0) {
        CRow& r = sh.row[s];
        r.M = big_m;
        r.log2s = log2s;
        r.ls = ls;
        r.c2 = c0 + log2s;
        r.cthr = mraw - fmaxf(fabsf(mraw) * 0x1p-20f, ro.qt * 0x1p-140f);
        r.B = bs;
        r.cB = cB;
        // raw rows: a group can pass the race bound (x ls - cB >= -24) only
        // if its largest logit reaches xB = (cB - 24) / ls, taken as (cB -
        // 24) T ln 2 and lowered by a relative 2^-18 (the roundings of ls,
        // of the product and of the fused multiply-add are below 2^-20)
        const float num = (cB - 24.0f) - fabsf(cB - 24.0f) * 0x1p-20f - 0x1p-16f;
        const float xb = num * (ro.qt * kLn2);
        r.xB = xb - fabsf(xb) * 0x1p-18f;
        r.qt = ro.qt;
        r.qy = ro.qy;
        r.qmode = ro.qmode;
        r.flags = (noisy ? kFNoisy : 0) | (topk && !hard ? kFTopk : 0) | (raw ? kFRaw : 0);
        r.bcol = bc;
        if (rank == 0) {
            RowRecord rec{};
            rec.M = big_m;
            rec.log2s = log2s;
            rec.lns = log2s * kLn2;
            rec.ls = ls;
            rec.c2 = r.c2;
            rec.thr = thr;
            rec.arg = arg_row;
            rec.cthr = r.cthr;
            rec.qt = ro.qt;
            rec.qy = ro.qy;
            rec.qmode = ro.qmode;
            rec.flags = r.flags;
            unsigned char* entry = p.rr + static_cast<int64_t>(ro.row) * p.rec_bytes;
            *reinterpret_cast<RowRecord*>(entry) = rec;
            *reinterpret_cast<SeedRec*>(entry + sizeof(RowRecord)) = SeedRec{bs, cB, bc, 0};
            if (stats) p.entropy[ro.row] = s_tot > 0.0f ? logf(s_tot) - w_tot / s_tot : 0.0f;
            if (p.out_m) {
                p.out_m[ro.row] = big_m;
                p.out_logs[ro.row] = rec.lns;
            }
            if (hard) {
                const int idx = atomicAdd(p.hard, 1);
                p.hard[kHardOffset + idx] = static_cast<int32_t>(ro.row);
            }
        }
    }
    return true;
}

// ------------------------------------------------------ phase B

// Probabilities of a whole chunk with aligned rows: 2^t rounded to nearest
// even, t = x ls - c2 (raw rows) or (s - M) log2(e) - log2 S. For bf16 the
// exponential is taken at t + 64 and scaled by 2^-64, so that fp32 subnormal
// results (which bf16 can hold down to 2^-133) are kept without the
// subnormal-keeping exponential; fp16 holds nothing below 2^-25, so the
// flushing one is exact there. -inf logits give 0.
template <bool BF16, bool RAW>
__device__ __forceinline__ void probs_full(const float4 (&v)[kCSlots], const CRow& r, const ScaledQuotient& sq,
                                           uint16_t* prow, int ct) {
    const float lift = BF16 ? 64.0f : 0.0f;
    const float2 l2 = make_float2(r.ls, r.ls);
    const float cp = r.c2 - lift;
    const float2 n2 = make_float2(-cp, -cp);
    const float2 d2 = make_float2(BF16 ? 0x1p-64f : 1.0f, BF16 ? 0x1p-64f : 1.0f);
    const FarBelow far(r.cthr, r.ls);  // exact rows only
#pragma unroll
    for (int i = 0; i < kCSlots; ++i) {
        const int f = i * kCompThreads + ct;
        float2 t01, t23;
        if (RAW) {
            t01 = __ffma2_rn(make_float2(v[i].x, v[i].y), l2, n2);
            t23 = __ffma2_rn(make_float2(v[i].z, v[i].w), l2, n2);
        } else {
            // (cthr is at most the row's raw max: a lower reference only
            // makes the far test more cautious)
            const float o = lift - r.log2s;
            const bool f0 = far(v[i].x), f1 = far(v[i].y), f2 = far(v[i].z), f3 = far(v[i].w);
            if (__any_sync(0xffffffffu, !(f0 && f1 && f2 && f3))) {
                t01 = make_float2(f0 ? kFarStandIn : fmaf(sq.exact(v[i].x) - r.M, kLog2e, o),
                                  f1 ? kFarStandIn : fmaf(sq.exact(v[i].y) - r.M, kLog2e, o));
                t23 = make_float2(f2 ? kFarStandIn : fmaf(sq.exact(v[i].z) - r.M, kLog2e, o),
                                  f3 ? kFarStandIn : fmaf(sq.exact(v[i].w) - r.M, kLog2e, o));
            } else {
                t01 = make_float2(kFarStandIn, kFarStandIn);
                t23 = t01;
            }
        }
        float2 e01 = make_float2(ex2_ftz(t01.x), ex2_ftz(t01.y));
        float2 e23 = make_float2(ex2_ftz(t23.x), ex2_ftz(t23.y));
        if (BF16) {
            e01 = __fmul2_rn(e01, d2);
            e23 = __fmul2_rn(e23, d2);
        }
        __stcs(reinterpret_cast<uint2*>(prow + 4 * f),
               make_uint2(pack2<BF16>(e01.x, e01.y), pack2<BF16>(e23.x, e23.y)));
    }
}

// Probabilities of a ragged chunk (fewer columns, or rows without aligned
// 8-byte stores): per-slot checks, the subnormal-keeping exponential.
template <bool BF16, bool RAW>
__device__ __forceinline__ void probs_ragged(const float4 (&v)[kCSlots], const CRow& r, const ScaledQuotient& sq,
                                             uint16_t* prow, bool vec, int ncols, int ct) {
#pragma unroll
    for (int i = 0; i < kCSlots; ++i) {
        const int f = i * kCompThreads + ct;
        if (4 * f >= ncols) continue;
        float pr[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float x = comp(v[i], q);
            const float tq = RAW                         ? fmaf(x, r.ls, -r.c2)
                             : FarBelow(r.cthr, r.ls)(x) ? kFarStandIn
                                                         : fmaf(sq.exact(x) - r.M, kLog2e, -r.log2s);
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

// The top-k candidates of a thread's slots in `smask` (slot i: bit i): the
// logits x >= thr, read again from the chunk, keyed by (exact value, lower
// column) into the CTA's list.
__device__ __noinline__ void topk_collect_chunk(uint32_t smask, const float4* chunk, int ct, int c0, int ncols,
                                                float thr, ScaledQuotient sq, int* count, uint64_t* kdst) {
    while (smask) {
        const int f = (__ffs(smask) - 1) * kCompThreads + ct;
        smask &= smask - 1;
        const float4 x4 = chunk[f];
        for (int q = 0; q < 4; ++q) {
            const float x = comp(x4, q);
            if (4 * f + q < ncols && x >= thr) {
                const int pos = atomicAdd(count, 1);
                if (pos < kTileKeys) kdst[pos] = topk_key(sq.exact(x), c0 + 4 * f + q);
            }
        }
    }
}

// One listed race group at float4 f of the chunk with its noise words nw:
// the group's largest e^(s - B) against the bound from its largest word
// (an element can only win if 1 - u <= -log u <= e^(s - B)), then element by
// element, and the few survivors rescored exactly against the best so far.
template <bool RAW>
__device__ __forceinline__ void race_group(const CRow& r, const ScaledQuotient& sq, const float4* chunk, int f,
                                           const uint4& nw, int c0, float& wb, int& wc) {
    const uint32_t wmax = max(max(nw.x, nw.y), max(nw.z, nw.w));
    const float4 x4 = chunk[f];
    const float mx = max4f(x4);
    const float emax = RAW ? ex2_ftz(fmaf(mx, r.ls, -r.cB)) : ex2_ftz(fmaf(sq.exact(mx) - r.B, kLog2e, kRaceSlack));
    if (one_minus_u_lower(wmax) <= emax) {
        const float4 e = race_e(x4, RAW, r.ls, SeedRec{r.B, r.cB, r.bcol, 0}, sq);
        uint32_t bits = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (one_minus_u_lower(word_of(nw, q)) <= comp(e, q)) bits |= 1u << q;
        if (bits) {
            const Best b2 = race_rescore(bits, x4, nw, c0 + 4 * f, r.bcol, sq, Best{wb, wc});
            wb = b2.s;
            wc = b2.c;
        }
    }
}

// One compute warp's share of phase B of a row; returns its result (valid
// on every lane). PD: 0 no probabilities, 1 bf16, 2 fp16.
template <int PD, bool RAW>
__device__ __forceinline__ WarpRes phase_b(const SplitParams& p, ClusterSmem& sh, const CRow& r,
                                           const float4* chunk, const RowSlot& ro, int c0, int ncols, int64_t t,
                                           int s, bool stats, int ct, int lane, int warp) {
    const ScaledQuotient sq{r.qt, r.qy, r.qmode};
    float4 v[kCSlots];
#pragma unroll
    for (int i = 0; i < kCSlots; ++i) v[i] = chunk[i * kCompThreads + ct];
    if (PD != 0 && stats) {
        uint16_t* prow = static_cast<uint16_t*>(p.probs) + static_cast<int64_t>(ro.row) * p.probs_row_stride + c0;
        if (r.M == -INFINITY) {
            // a row that is -inf everywhere: NaN
            const uint16_t code = static_cast<uint16_t>(pack2<PD == 1>(NAN, NAN));
            for (int cidx = ct; cidx < ncols; cidx += kCompThreads) prow[cidx] = code;
        } else if (p.probs_vec && ncols == kCChunkMax) {
            probs_full<PD == 1, RAW>(v, r, sq, prow, ct);
        } else {
            probs_ragged<PD == 1, RAW>(v, r, sq, prow, p.probs_vec != 0, ncols, ct);
        }
    }
    float m4[kCSlots];
#pragma unroll
    for (int i = 0; i < kCSlots; ++i) m4[i] = max4f(v[i]);
    float mthr = max3(m4[0], m4[1], m4[2]);
    mthr = max3(mthr, m4[3], m4[4]);
    mthr = max3(mthr, m4[5], m4[6]);
    mthr = fmaxf(mthr, m4[7]);

    // argmax ties: logits below the raw max whose exact quotient is M (rare)
    int acand = INT_MAX;
    if (stats && r.M != -INFINITY && mthr >= r.cthr) {
        uint32_t am = 0;
#pragma unroll
        for (int i = 0; i < kCSlots; ++i) am |= (m4[i] >= r.cthr ? 1u : 0u) << i;
#pragma unroll 1
        while (am && acand == INT_MAX) {
            const int f = (__ffs(am) - 1) * kCompThreads + ct;
            am &= am - 1;
            const float4 x4 = chunk[f];
#pragma unroll 1
            for (int q = 0; q < 4; ++q) {
                const float x = comp(x4, q);
                if (4 * f + q < ncols && x >= r.cthr && sq.exact(x) == r.M) {
                    acand = c0 + 4 * f + q;
                    break;
                }
            }
        }
    }

    // the race: groups whose largest e^(s - B) can reach 2^-24, listed
    // warp-wide and shared out one Philox call per lane
    float wb = r.B;
    int wc = r.bcol;
    if (r.flags & kFNoisy) {
        uint32_t pass = 0;
        if (RAW) {
#pragma unroll
            for (int i = 0; i < kCSlots; ++i)
                if (m4[i] >= r.xB) pass |= 1u << i;
        } else {
#pragma unroll
            for (int i = 0; i < kCSlots; ++i)
                if (fmaf(sq.exact(m4[i]) - r.B, kLog2e, kRaceSlack) >= -24.0f) pass |= 1u << i;
        }
        if (__any_sync(0xffffffffu, pass != 0)) {
            const uint32_t lt = lanemask_lt();
            int total = 0;
            uint16_t* list = sh.race_at[warp];
#pragma unroll
            for (int i = 0; i < kCSlots; ++i) {
                const bool on = (pass >> i) & 1u;
                const uint32_t bl = __ballot_sync(0xffffffffu, on);
                if (on) list[total + __popc(bl & lt)] = static_cast<uint16_t>(i * kCompThreads + ct);
                total += __popc(bl);
            }
            __syncwarp();
            const uint32_t g0 = static_cast<uint32_t>(c0 >> 2);
            const RowNoise rn = row_noise(p.rk[0], static_cast<uint64_t>(p.row0 + ro.row));
            for (int m = lane; m < total; m += 32) {
                const int f = list[m];
                const uint4 nw = noise_folded(p.rk[0], rn, g0 + static_cast<uint32_t>(f));
                race_group<RAW>(r, sq, chunk, f, nw, c0, wb, wc);
            }
        }
    }

    // top-k candidates x >= thr (rare: the slots reaching it)
    if ((r.flags & kFTopk) && mthr >= r.thr) {
        uint32_t km = 0;
#pragma unroll
        for (int i = 0; i < kCSlots; ++i) km |= (m4[i] >= r.thr ? 1u : 0u) << i;
        if (km) topk_collect_chunk(km, chunk, ct, c0, ncols, r.thr, sq, &sh.tile_nk[s], p.keys + t * kTileKeys);
    }
    warp_best(wb, wc);
    return WarpRes{wb, wc, warp_min_nonneg(acand), 0};
}

// ------------------------------------------------------ the kernel

// Grid: clusters of C CTAs (C = the cluster size of the launch), one CTA per
// SM; cluster q takes list entries list_begin + q, + nclusters, ... Every CTA
// owns columns [rank * chunk_cols, min(V, (rank + 1) * chunk_cols)) of each
// of its rows.
template <int PD>
__global__ void __launch_bounds__(kCThreads, 1) split_cluster(const __grid_constant__ SplitParams p,
                                                             const ClusterShape cs) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    extern __shared__ __align__(128) unsigned char smem_dyn[];
    float4* buf = reinterpret_cast<float4*>(smem_dyn);
    __shared__ __align__(16) ClusterSmem sh;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const uint32_t rank = cta_rank();
    const uint32_t C = cta_count();
    const int ncl = static_cast<int>(cluster_total());
    const int c0 = static_cast<int>(rank) * cs.chunk_cols;
    const int ncols = min(max(p.vocab - c0, 0), cs.chunk_cols);
    const bool stats = p.stats != 0;
    const int lend = list_end(p);
    const int li0 = list_begin(p) + static_cast<int>(cluster_index());
    const int T = li0 < lend ? (lend - li0 + ncl - 1) / ncl : 0;  // rows of this cluster

    // the buffers past this CTA's columns read as -inf (never copied into)
    for (int b = 0; b < kCBufs; ++b)
        for (int f = (ncols >> 2) + tid; f < kCChunkF4; f += kCThreads)
            buf[b * kCChunkF4 + f] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    if (tid == 0) {
        for (int b = 0; b < kCBufs; ++b) {
            mbar_init(&sh.full[b], 1);
            sh.issued[b] = -1;
        }
        for (int s = 0; s < kCPartSlots; ++s) mbar_init(&sh.part_full[s], 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sh.adone[s], kCompWarps);
            mbar_init(&sh.bdone[s], kCompWarps);
            mbar_init(&sh.recrdy[s], 1);
            mbar_init(&sh.cand_done[s], 1);
            mbar_init(&sh.thr_done[s], 1);
            sh.tile_nk[s] = 0;
        }
        sh.abort = 0;
        fence_barrier_init();
    }
    __syncthreads();
    cluster_sync_all();  // every CTA's barriers are set before any push

    if (warp == kFeedWarp) {
        // ================================ the feed warp: the row ring, the
        // copies, and the per-tile records after phase B
        fill_ring(p, sh, li0, ncl, T, 0, lane);
        fill_ring(p, sh, li0, ncl, T, 32, lane);
        __syncwarp();
        if (lane == 0)
            for (int b = 0; b < kCBufs && b < T; ++b) issue_row(p, sh, buf, b, b, c0, ncols);
        for (int u = 0; u < T; ++u) {
            const int s = u & 1;
            if (!__all_sync(0xffffffffu,
                            wait_phase<false>(&sh.bdone[s], static_cast<uint32_t>((u >> 1) & 1), &sh.abort))) {
                if (lane == 0) give_up(sh, p.err);
                break;
            }
            float b = lane < kCompWarps ? sh.wres[s][lane].b : -INFINITY;
            int bc = lane < kCompWarps ? sh.wres[s][lane].c : INT_MAX;
            warp_best(b, bc);
            const int a = warp_min_nonneg(lane < kCompWarps ? sh.wres[s][lane].a : INT_MAX);
            const int t = u + kCBufs;  // the row that goes into the freed buffer
            // rows t + 32 .. t + 63 into the ring (their slots held rows long done)
            if (t < T && (t & 31) == 0 && t >= 32) fill_ring(p, sh, li0, ncl, T, t + 32, lane);
            __syncwarp();
            if (lane == 0) {
                // the CTA is tile `rank` of the row's G = tiles_per_row
                // records (G >= C: the two passes' tiles of 8192 columns);
                // tile rank + C, past the cluster's C, is written empty
                const int G = p.tiles_per_row;
                const int64_t tt = static_cast<int64_t>(li0 + u * ncl) * G + rank;
                p.tb[tt] = TileSeed{b, bc};
                p.te[tt] = TileEnd{sh.ring[u % kCRing].kept && p.k > 0 ? sh.tile_nk[s] : 0, a};
                if (static_cast<int>(rank + C) < G) {
                    p.tb[tt + C] = TileSeed{-INFINITY, INT_MAX};
                    p.te[tt + C] = TileEnd{0, INT_MAX};
                }
                sh.tile_nk[s] = 0;
                if (t < T) {
                    fence_proxy_async_smem();
                    issue_row(p, sh, buf, u % kCBufs, t, c0, ncols);
                }
            }
            __syncwarp();
        }
        if (lane == 0 && sh.abort) {
            // copies still in flight land before the shared memory is released
            for (int b = 0; b < kCBufs; ++b)
                if (sh.issued[b] >= 0)
                    mbar_wait_bounded(&sh.full[b], static_cast<uint32_t>((sh.issued[b] / kCBufs) & 1));
        }
    } else if (warp == kMergeWarp) {
        // ================================ the merge warp: the CTA's part of
        // each row, pushed to the cluster; the merge of the C parts
        for (int t = 0; t < T; ++t) {
            const int s = t & 1;
            const uint32_t par = static_cast<uint32_t>((t >> 1) & 1);
            if (!__all_sync(0xffffffffu, wait_phase<false>(&sh.adone[s], par, &sh.abort))) {
                if (lane == 0) give_up(sh, p.err);
                break;
            }
            const RowSlot ro = sh.ring[t % kCRing];
            const int ps = t % kCPartSlots;
            const uint32_t ppar = static_cast<uint32_t>((t / kCPartSlots) & 1);
            const uint32_t nw = part_words(ro.kept && p.k > 0, cs.top_m);
            // the slot's phase for row t: C parts of nw words (parts that
            // landed already count against it; the arrival completes it)
            if (lane == 0) mbar_arrive_expect_tx(&sh.part_full[ps], nw * 16u * C);
            make_part(p, sh, ro, ncols, c0, cs.top_m, s, rank, C, lane);
            if (!__all_sync(0xffffffffu, wait_phase<false>(&sh.cand_done[s], par, &sh.abort))) {
                if (lane == 0) give_up(sh, p.err);
                break;
            }
            if (lane == 0) {
                sh.mine.bs = sh.cand_s[s];
                sh.mine.bc = sh.cand_c[s];
            }
            push_part(sh, ps, rank, C, nw, lane);
            if (!__all_sync(0xffffffffu, wait_phase<true>(&sh.part_full[ps], ppar, &sh.abort)) ||
                !merge_parts(p, sh, ro, stats, s, static_cast<int>(par), ps, rank, C, lane)) {
                if (lane == 0) give_up(sh, p.err);
                break;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.recrdy[s]);
        }
    } else if (warp == kNoiseWarp) {
        // ================================ the noise warp: each row's Gumbel
        // candidates (for B), then its top-k threshold once the parts land
        for (int t = 0; t < T; ++t) {
            const int s = t & 1;
            const uint32_t par = static_cast<uint32_t>((t >> 1) & 1);
            if (!__all_sync(0xffffffffu, wait_phase<false>(&sh.adone[s], par, &sh.abort))) {
                if (lane == 0) give_up(sh, p.err);
                break;
            }
            const RowSlot ro = sh.ring[t % kCRing];
            score_candidates(p, sh, ro, stats, s, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.cand_done[s]);
            // (every row takes one phase of thr_done, so that its parity
            // stays that of the row, whether the row wants a threshold or not)
            if (ro.kept && p.k > 0) {
                const int ps = t % kCPartSlots;
                if (!__all_sync(0xffffffffu,
                                try_wait_parts(sh, ps, static_cast<uint32_t>((t / kCPartSlots) & 1)))) {
                    if (lane == 0) give_up(sh, p.err);
                    break;
                }
                row_threshold(p, sh, ro, cs.top_m, s, ps, C, lane);
                __syncwarp();
            }
            if (lane == 0) mbar_arrive(&sh.thr_done[s]);
        }
    } else {
        // ================================ the compute warps
        const int ct = tid - 32 * kCtlWarps;  // 0 .. 511
        const int cw = warp - kCtlWarps;      // 0 .. 15
        for (int t = 0; t <= T; ++t) {
            if (t < T) {
                const int b = t % kCBufs;
                if (!__all_sync(0xffffffffu,
                                wait_phase<false>(&sh.full[b], static_cast<uint32_t>((t / kCBufs) & 1), &sh.abort))) {
                    if (lane == 0) give_up(sh, p.err);
                    break;
                }
                const RowSlot& ro = sh.ring[t % kCRing];
                const ScaledQuotient sq{ro.qt, ro.qy, ro.qmode};
                const WarpPart wp = phase_a(buf + b * kCChunkF4, sq, c0, ct, stats);
                if (lane == 0) {
                    sh.wparts[t & 1][cw] = wp;
                    mbar_arrive(&sh.adone[t & 1]);
                }
            }
            if (t >= 1) {
                const int u = t - 1;
                const int s = u & 1;
                if (!__all_sync(0xffffffffu,
                                wait_phase<false>(&sh.recrdy[s], static_cast<uint32_t>((u >> 1) & 1), &sh.abort))) {
                    if (lane == 0) give_up(sh, p.err);
                    break;
                }
                const CRow r = sh.row[s];
                const RowSlot ro = sh.ring[u % kCRing];
                const int64_t tt = static_cast<int64_t>(li0 + u * ncl) * p.tiles_per_row + rank;
                const float4* chunk = buf + (u % kCBufs) * kCChunkF4;
                const WarpRes wr =
                    (r.flags & kFRaw)
                        ? phase_b<PD, true>(p, sh, r, chunk, ro, c0, ncols, tt, s, stats, ct, lane, cw)
                        : phase_b<PD, false>(p, sh, r, chunk, ro, c0, ncols, tt, s, stats, ct, lane, cw);
                if (lane == 0) {
                    sh.wres[s][cw] = wr;
                    mbar_arrive(&sh.bdone[s]);
                }
            }
        }
    }
    asm volatile("griddepcontrol.launch_dependents;");
}

}  // namespace

bool cluster_plan(int64_t rows, int64_t vocab, int32_t k, int32_t n_seeds, bool aligned16, ClusterShape* out,
                  int* cluster_size) {
    if (rows <= 0 || vocab < 1 || vocab > static_cast<int64_t>(kCMaxCluster) * kCChunkMax) return false;
    if (!aligned16 || (vocab & 3) != 0 || n_seeds != 1 || k > kSplitMaxK) return false;
    const int V = static_cast<int>(vocab);
    const int C = (V + kCChunkMax - 1) / kCChunkMax;
    const int f4 = V / 4;
    const int chunk = 4 * ((f4 + C - 1) / C);
    ClusterShape cs{};
    cs.chunk_cols = chunk;
    cs.pieces = 1;
    // each CTA publishes its largest group maxima: enough that about 2k of
    // them reach the merge (the threshold's quality)
    const int m = k > 0 ? (2 * k + C - 1) / C : 1;
    cs.top_m = m > kCGroups ? kCGroups : m;
    *out = cs;
    *cluster_size = C;
    return true;
}

namespace {

// The launch configuration of the cluster kernel for a probability dtype.
void (*cluster_kernel(int probs_dtype))(SplitParams, ClusterShape) {
    return probs_dtype == 1 ? split_cluster<1> : probs_dtype == 2 ? split_cluster<2> : split_cluster<0>;
}

bool cluster_config(void (*kernel)(SplitParams, ClusterShape), int C, cudaStream_t stream,
                    cudaLaunchAttribute (&attr)[3], cudaLaunchConfig_t& cfg) {
    const size_t smem = static_cast<size_t>(kCBufs) * kCChunkF4 * sizeof(float4);
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
            cudaSuccess ||
        cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
        return false;
    cfg = cudaLaunchConfig_t{};
    cfg.blockDim = dim3(kCThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(C);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    // the device's highest launch priority: when the two passes run beside
    // it on the SMs the clusters leave, the clusters are placed first
    int least = 0, greatest = 0;
    if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) return false;
    attr[2].id = cudaLaunchAttributePriority;
    attr[2].val.priority = greatest;
    cfg.attrs = attr;
    cfg.numAttrs = 3;
    cfg.gridDim = dim3(static_cast<unsigned>(C));
    return true;
}

}  // namespace

int cluster_active(int probs_dtype, int C) {
    void (*kernel)(SplitParams, ClusterShape) = cluster_kernel(probs_dtype);
    cudaLaunchAttribute attr[3];
    cudaLaunchConfig_t cfg;
    if (!cluster_config(kernel, C, nullptr, attr, cfg)) return 0;
    int active = 0;
    if (cudaOccupancyMaxActiveClusters(&active, kernel, &cfg) != cudaSuccess) return 0;
    return active;
}

drs_status cluster_launch(const SplitParams& p, const ClusterShape& cs, int C, int64_t rows,
                          cudaStream_t stream) {
    void (*kernel)(SplitParams, ClusterShape) = cluster_kernel(p.probs_dtype);
    cudaLaunchAttribute attr[3];
    cudaLaunchConfig_t cfg;
    if (!cluster_config(kernel, C, stream, attr, cfg)) return DRS_ERR_CUDA;
    // as many clusters as can be resident at once (each loops over rows),
    // no more than rows
    int active = 0;
    if (cudaOccupancyMaxActiveClusters(&active, kernel, &cfg) != cudaSuccess || active < 1) return DRS_ERR_CUDA;
    const int64_t ncl = rows < active ? rows : active;
    cfg.gridDim = dim3(static_cast<unsigned>(ncl * C));
    return cudaLaunchKernelEx(&cfg, kernel, p, cs) == cudaSuccess ? DRS_OK : DRS_ERR_CUDA;
}

}  // namespace rs
}  // namespace drs
