// row_cluster.cu -- the row statistics with ONE read of the logits (page
// "vllm.model_executor.models.diffusion_gemma_sampler": the module docstring's
// single read with an online max and sum, the noise drawn inline and one write
// of the probabilities; sample_row_stats_reference for what is computed).
//
// A row is split over the C CTAs of a thread-block cluster, each owning a
// contiguous chunk of at most 16384 columns (64 KiB), which stays in its
// shared memory from the bulk copy (TMA) that brings it in until the
// probabilities have been written from it. Per row and CTA:
//   phase A  per warp and piece (8192 columns), the raw max and its lowest
//            column, S = sum e^(s - m) and W = sum e^(s - m)(s - m) (as
//            pass 1 of the two-pass kernels: raw-domain exponentials while
//            |m| < 256, exact quotients beyond);
//   part     warp 0 combines the warps into the CTA's part (m, S, W, raw max
//            and column, the best Gumbel-max score of the warps' argmax
//            elements, the CTA's largest group maxima) and pushes it into
//            every CTA of the cluster (st.async into distributed shared
//            memory, completing on each receiver's mbarrier);
//   merge    every CTA waits for the C parts (a bounded wait) and merges them
//            the same way: the row's M, S, W, argmax column, B, the top-k
//            threshold (the k-th largest of the parts' group maxima);
//   phase B  per warp and piece, from shared memory: the probabilities, the
//            argmax ties, the pruned Gumbel race against B, the top-k
//            candidates; as each piece is done the next row's copy into it
//            starts.
// The CTA's race winner, argmax tie and candidates go to the same per-tile
// records the two-pass kernels write (a CTA is one tile of its row), and the
// finish kernel of row_split.cu reduces them.
//
// HBM traffic: every logit read once, every probability written once.
#include "row_common.cuh"

namespace drs {
namespace rs {
namespace {

constexpr int kCPieceF4 = kStageF4;     // 2048 float4 per piece: 8 per thread
constexpr int kCPieceCols = kTileCols;  // 8192 columns
constexpr int kCMaxPieces = 2;
constexpr int kCMaxCluster = 16;
constexpr int kCChunkMax = kCMaxPieces * kCPieceCols;  // 16384 columns per CTA
constexpr int kCGroups = kSWarps * kCMaxPieces;        // warp-piece groups per CTA

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
constexpr uint32_t kCPartWords = sizeof(CPart) / 16;

// The merged row as phase B uses it.
struct CRow {
    float M, log2s, ls, c2, thr, cthr, B, cB, xB;
    float qt, qy;
    int qmode, flags, bcol, pad;
};

struct ClusterSmem {
    uint64_t piece_full[kCMaxPieces];  // the chunk's pieces landed (TMA)
    uint64_t part_full[2];             // the C parts of a row landed (by row parity)
    int piece_count[kCMaxPieces];      // warps done with a piece in phase B
    int last_issue[kCMaxPieces];       // row iteration of the last copy into a piece
    int abort;
    int tile_nk;                       // top-k candidates of the CTA for the row
    CPart part[2][kCMaxCluster];
    CPart mine;
    WarpPart wparts[kCMaxPieces][kSWarps];
    CRow row;
    float best_s[kSWarps];
    int best_c[kSWarps];
    int best_a[kSWarps];
    uint16_t race_at[kSWarps][kSVec4 * 32];
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

// Phase-parity wait on an mbarrier completed by other CTAs' pushes
// (acquire at cluster scope), bounded like mbar_wait_bounded.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
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
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait_cluster(bar, parity, 1000u)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait_cluster(bar, parity, 100000u)) return true;
        if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// ------------------------------------------------------ loading

// Columns of this CTA in piece j.
__device__ __forceinline__ int piece_cols(int ncols, int j) {
    return min(max(ncols - j * kCPieceCols, 0), kCPieceCols);
}

// Issue the copy of piece j of list entry li (row iteration `it` of the
// cluster) into the buffer; a piece without columns completes with a plain
// arrival.
__device__ __forceinline__ void issue_piece(const SplitParams& p, ClusterSmem& sh, float4* buf, int j,
                                            int li, int it, int c0, int ncols) {
    sh.last_issue[j] = it;
    if (p.fault && it == 0 && j == 0 && blockIdx.x == 0) {
        // the test hook: this piece never lands, the waits on it run out
        sh.last_issue[j] = -1;
        return;
    }
    const int n = piece_cols(ncols, j);
    if (n == 0) {
        mbar_arrive(&sh.piece_full[j]);
        return;
    }
    const int row = p.list1[li];
    const int64_t lrow = p.map_row ? p.map_row[row] : row;
    const uint32_t bytes = static_cast<uint32_t>(n) * 4u;
    mbar_arrive_expect_tx(&sh.piece_full[j], bytes);
    tma_load_1d(buf + j * kCPieceF4, p.logits + lrow * p.row_stride + c0 + j * kCPieceCols, bytes,
                &sh.piece_full[j]);
}

// ------------------------------------------------------ phase A

// S = sum 2^t and W = ln2 * sum 2^t t, t = x * ls - cref, over a thread's 32
// logits, two at a time; with CLAMP, t is kept finite (a -inf logit gives
// e = 0 and e * t = 0 instead of NaN).
template <bool CLAMP>
__device__ __forceinline__ void sums2(const float4 (&v)[kSVec4], float ls, float cref, float& sw, float& ww) {
    const float2 l2 = make_float2(ls, ls), n2 = make_float2(-cref, -cref);
    float2 sa = make_float2(0.0f, 0.0f), sb = sa, wa = sa, wb = sa;
#pragma unroll
    for (int i = 0; i < kSVec4; ++i) {
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

// One warp's share of a piece: the raw max M_w of its 1024 columns and the
// lowest column holding it, S_w and W_w relative to it (raw domain while
// |M_w| < 256 for sure, else from exact quotients).
__device__ __forceinline__ WarpPart phase_a(const float4* piece, const ScaledQuotient& sq, int col0, int tid,
                                            bool want_arg) {
    float4 v[kSVec4];
    float mt = -INFINITY;
#pragma unroll
    for (int i = 0; i < kSVec4; ++i) {
        v[i] = piece[i * kSThreads + tid];
        mt = max3(mt, v[i].x, v[i].y);
        mt = max3(mt, v[i].z, v[i].w);
    }
    const float mxw = warp_max_f(mt);
    if (mxw == -INFINITY) return WarpPart{0.0f, 0.0f, 0.0f, -INFINITY, INT_MAX};
    int arg_t = INT_MAX;
    if (want_arg && mt == mxw) {
        int i0 = 0;
#pragma unroll
        for (int i = kSVec4 - 1; i >= 0; --i)
            if (max4f(v[i]) == mxw) i0 = i;
        const int f = i0 * kSThreads + tid;
        const float4 x4 = piece[f];
        const int q = x4.x == mxw ? 0 : x4.y == mxw ? 1 : x4.z == mxw ? 2 : 3;
        arg_t = col0 + 4 * f + q;
    }
    const int aw = want_arg ? warp_min_nonneg(arg_t) : INT_MAX;
    const bool raw = fabsf(mxw * sq.y) < kRawLimit - 1.0f;
    float lscale, cref;
    if (raw) {
        lscale = kLog2e * sq.y;
        cref = mxw * lscale;
    } else {
        const float mw = sq.exact(mxw);
#pragma unroll
        for (int i = 0; i < kSVec4; ++i) {
            v[i].x = sq.exact(v[i].x) - mw;
            v[i].y = sq.exact(v[i].y) - mw;
            v[i].z = sq.exact(v[i].z) - mw;
            v[i].w = sq.exact(v[i].w) - mw;
        }
        lscale = kLog2e;
        cref = 0.0f;
    }
    float sw, ww;
    sums2<false>(v, lscale, cref, sw, ww);
    if (isnan(ww)) sums2<true>(v, lscale, cref, sw, ww);
    return WarpPart{0.0f, sw, ww, mxw, aw};
}

// Warp 0: the CTA's part from the warp parts (lane l < 8 P holds piece l / 8,
// warp l % 8), into sh.mine, then pushed into slot `s` of every CTA.
__device__ __forceinline__ void make_part(const SplitParams& p, ClusterSmem& sh, const ScaledQuotient& sq,
                                          uint64_t grow, bool noisy, int pieces, int ncols, int c0, int top_m,
                                          int s, uint32_t rank, uint32_t C, int lane) {
    const int nparts = pieces * kSWarps;
    WarpPart wp = lane < nparts ? sh.wparts[lane / kSWarps][lane % kSWarps]
                                : WarpPart{0.0f, 0.0f, 0.0f, -INFINITY, INT_MAX};
    const bool present = lane < nparts && (lane / kSWarps) * kCPieceCols + (lane % kSWarps) * 128 < ncols;
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
    // the Gumbel-max score of each warp's argmax element (its exact
    // quotient is M_w)
    float bs = -INFINITY;
    int bc = INT_MAX;
    if (noisy && wp.arg != INT_MAX) {
        const uint4 nw = noise_group(p.rk[0], grow, static_cast<uint32_t>(wp.arg >> 2));
        bs = wp.m + gumbel_of_bits(word_of(nw, wp.arg & 3));
        bc = wp.arg;
    }
    warp_best(bs, bc);
    // the CTA's top_m group maxima, descending (absent groups are 0, below
    // every value; -inf is kOrdNegInf)
    uint32_t key = present ? ord32(wp.xmax) : 0u;
    uint32_t mine = 0;
    int ng = 0;
    for (int r = 0; r < top_m; ++r) {
        uint32_t top;
        asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(top) : "r"(key));
        if (top == 0) break;
        if (lane == r) mine = top;
        ++ng;
        const uint32_t holders = __ballot_sync(0xffffffffu, key == top);
        if (lane == __ffs(holders) - 1) key = 0;
    }
    if (lane < kCGroups) sh.mine.gm[lane] = mine;
    if (lane == 0) {
        sh.mine.m = mc;
        sh.mine.s = s_c;
        sh.mine.w = w_c;
        sh.mine.xmax = xm;
        sh.mine.arg = a_c;
        sh.mine.bs = bs;
        sh.mine.bc = bc;
        sh.mine.ng = ng;
    }
    __syncwarp();
    const uint4* src = reinterpret_cast<const uint4*>(&sh.mine);
    const uint32_t dst = smem_u32(&sh.part[s][rank]);
    const uint32_t bar = smem_u32(&sh.part_full[s]);
    for (uint32_t idx = lane; idx < kCPartWords * C; idx += 32) {
        const uint32_t d = idx / kCPartWords;
        const uint32_t q = idx - d * kCPartWords;
        push16(map_to_rank(dst + 16u * q, d), src[q], map_to_rank(bar, d));
    }
}

// Warp 0: the row from the C parts in slot s (NU: group maxima per lane in
// the threshold's selection). Every CTA computes the same; CTA 0 of the
// cluster also writes the row's record for the finish kernel, the entropy,
// the stash's max and log S, and rows without a threshold on the hard list.
template <int NU>
__device__ __forceinline__ void merge_parts(const SplitParams& p, ClusterSmem& sh, const RowTemp& rt, int64_t row,
                                            bool stats, bool topk, int top_m, int s, uint32_t rank, uint32_t C,
                                            int lane) {
    const CPart* pr = sh.part[s];
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

    float thr = -INFINITY;
    bool hard = false;
    if (topk) {
        // the k-th largest of the parts' group maxima: k rounds of a warp
        // max, each removing one occurrence (k distinct elements reach it,
        // so the row's top k all do)
        const int n = static_cast<int>(C) * top_m;
        uint32_t o[NU];
#pragma unroll
        for (int u = 0; u < NU; ++u) {
            const int idx = lane + 32 * u;
            const int c = idx / top_m;
            o[u] = idx < n ? pr[c].gm[idx - c * top_m] : 0u;
        }
        uint32_t kth = 0;
        for (int rd = 0; rd < p.k; ++rd) {
            uint32_t lm = 0;
#pragma unroll
            for (int u = 0; u < NU; ++u) lm = max(lm, o[u]);
            uint32_t top;
            asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(top) : "r"(lm));
            kth = top;
            if (top == 0) break;
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
    const bool noisy = stats && rt.temp > 0.0f && big_m != -INFINITY;
    const float ls = kLog2e * rt.qy;
    const float c0 = mraw * ls;
    const float log2s = s_tot > 0.0f ? log2f(s_tot) : 0.0f;
    const bool raw = !(fabsf(big_m) >= kRawLimit);
    const float cB = (c0 + (bs - big_m) * kLog2e) - kRaceSlack;
    if (lane == 0) {
        CRow& r = sh.row;
        r.M = big_m;
        r.log2s = log2s;
        r.ls = ls;
        r.c2 = c0 + log2s;
        r.thr = thr;
        r.cthr = mraw - fmaxf(fabsf(mraw) * 0x1p-20f, rt.qt * 0x1p-140f);
        r.B = bs;
        r.cB = cB;
        // raw rows: a group can pass the race bound (x ls - cB >= -24) only
        // if its largest logit reaches xB (lowered by a relative 2^-20 for
        // the roundings of the quotient and of the fused multiply-add)
        const float xb = __fdiv_rn((cB - 24.0f) - fabsf(cB - 24.0f) * 0x1p-20f - 0x1p-16f, ls);
        r.xB = xb - fabsf(xb) * 0x1p-20f;
        r.qt = rt.qt;
        r.qy = rt.qy;
        r.qmode = rt.qmode;
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
            rec.qt = rt.qt;
            rec.qy = rt.qy;
            rec.qmode = rt.qmode;
            rec.flags = r.flags;
            unsigned char* entry = p.rr + row * p.rec_bytes;
            *reinterpret_cast<RowRecord*>(entry) = rec;
            *reinterpret_cast<SeedRec*>(entry + sizeof(RowRecord)) = SeedRec{bs, cB, bc, 0};
            if (stats) p.entropy[row] = s_tot > 0.0f ? logf(s_tot) - w_tot / s_tot : 0.0f;
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
}

// ------------------------------------------------------ phase B

// Probabilities of a piece with aligned rows and all 8192 columns present:
// 2^t rounded to nearest even, t = x ls - c2 (raw rows) or (s - M) log2(e)
// - log2 S. For bf16 the exponential is taken at t + 64 and scaled by 2^-64,
// so that fp32 subnormal results (which bf16 can hold down to 2^-133) are
// kept without the subnormal-keeping exponential; fp16 holds nothing below
// 2^-25, so the flushing one is exact there. -inf logits give 0.
template <bool BF16, bool RAW>
__device__ __forceinline__ void probs_full(const float4 (&v)[kSVec4], const CRow& r, const ScaledQuotient& sq,
                                           uint16_t* prow, int tid) {
    const float lift = BF16 ? 64.0f : 0.0f;
    const float2 l2 = make_float2(r.ls, r.ls);
    const float cp = r.c2 - lift;
    const float2 n2 = make_float2(-cp, -cp);
    const float2 d2 = make_float2(BF16 ? 0x1p-64f : 1.0f, BF16 ? 0x1p-64f : 1.0f);
#pragma unroll
    for (int i = 0; i < kSVec4; ++i) {
        const int f = i * kSThreads + tid;
        float2 t01, t23;
        if (RAW) {
            t01 = __ffma2_rn(make_float2(v[i].x, v[i].y), l2, n2);
            t23 = __ffma2_rn(make_float2(v[i].z, v[i].w), l2, n2);
        } else {
            const float o = lift - r.log2s;
            t01 = make_float2(fmaf(sq.exact(v[i].x) - r.M, kLog2e, o), fmaf(sq.exact(v[i].y) - r.M, kLog2e, o));
            t23 = make_float2(fmaf(sq.exact(v[i].z) - r.M, kLog2e, o), fmaf(sq.exact(v[i].w) - r.M, kLog2e, o));
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

// Probabilities of a ragged piece (fewer columns, or rows without aligned
// 8-byte stores): per-slot checks, the subnormal-keeping exponential.
template <bool BF16, bool RAW>
__device__ __forceinline__ void probs_ragged(const float4 (&v)[kSVec4], const CRow& r, const ScaledQuotient& sq,
                                             uint16_t* prow, bool vec, int ncols, int tid) {
#pragma unroll
    for (int i = 0; i < kSVec4; ++i) {
        const int f = i * kSThreads + tid;
        if (4 * f >= ncols) continue;
        float pr[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float x = comp(v[i], q);
            const float tq = RAW ? fmaf(x, r.ls, -r.c2) : fmaf(sq.exact(x) - r.M, kLog2e, -r.log2s);
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

// The per-lane state phase B carries over a row's pieces.
struct LaneBest {
    float wb;   // best race score so far
    int wc;     // its column
    int acand;  // lowest column below the raw max whose exact quotient is M
};

// One warp's share of a piece in phase B. PD: 0 no probabilities, 1 bf16,
// 2 fp16.
template <int PD, bool RAW>
__device__ __forceinline__ void phase_b(const SplitParams& p, ClusterSmem& sh, const CRow& r,
                                        const ScaledQuotient& sq, const float4* piece, uint64_t grow, int64_t row,
                                        int col0, int ncols, int64_t t, bool stats, int tid, int lane, int warp,
                                        LaneBest& lb) {
    float4 v[kSVec4];
#pragma unroll
    for (int i = 0; i < kSVec4; ++i) v[i] = piece[i * kSThreads + tid];
    if (PD != 0 && stats) {
        uint16_t* prow = static_cast<uint16_t*>(p.probs) + row * p.probs_row_stride + col0;
        if (r.M == -INFINITY) {
            // a row that is -inf everywhere: NaN
            const uint16_t code = static_cast<uint16_t>(pack2<PD == 1>(NAN, NAN));
            for (int cidx = tid; cidx < ncols; cidx += kSThreads) prow[cidx] = code;
        } else if (p.probs_vec && ncols == kCPieceCols) {
            probs_full<PD == 1, RAW>(v, r, sq, prow, tid);
        } else {
            probs_ragged<PD == 1, RAW>(v, r, sq, prow, p.probs_vec != 0, ncols, tid);
        }
    }
    float m4[kSVec4];
#pragma unroll
    for (int i = 0; i < kSVec4; ++i) m4[i] = max4f(v[i]);
    float mthr = max3(m4[0], m4[1], m4[2]);
    mthr = max3(mthr, m4[3], m4[4]);
    mthr = max3(mthr, m4[5], m4[6]);
    mthr = fmaxf(mthr, m4[7]);

    // argmax ties: logits below the raw max whose exact quotient is M (rare)
    if (stats && r.M != -INFINITY && mthr >= r.cthr && lb.acand == INT_MAX) {
        uint32_t am = 0;
#pragma unroll
        for (int i = 0; i < kSVec4; ++i) am |= (m4[i] >= r.cthr ? 1u : 0u) << i;
#pragma unroll 1
        while (am && lb.acand == INT_MAX) {
            const int f = (__ffs(am) - 1) * kSThreads + tid;
            am &= am - 1;
            const float4 x4 = piece[f];
#pragma unroll 1
            for (int q = 0; q < 4; ++q) {
                const float x = comp(x4, q);
                if (4 * f + q < ncols && x >= r.cthr && sq.exact(x) == r.M) {
                    lb.acand = col0 + 4 * f + q;
                    break;
                }
            }
        }
    }

    // the race: groups whose largest e^(s - B) can reach 2^-24, listed
    // warp-wide and shared out one Philox call per lane
    if (r.flags & kFNoisy) {
        uint32_t pass = 0;
        if (RAW) {
#pragma unroll
            for (int i = 0; i < kSVec4; ++i)
                if (m4[i] >= r.xB) pass |= 1u << i;
        } else {
#pragma unroll
            for (int i = 0; i < kSVec4; ++i)
                if (fmaf(sq.exact(m4[i]) - r.B, kLog2e, kRaceSlack) >= -24.0f) pass |= 1u << i;
        }
        if (__any_sync(0xffffffffu, pass != 0)) {
            const uint32_t lt = lanemask_lt();
            int total = 0;
            uint16_t* list = sh.race_at[warp];
#pragma unroll
            for (int i = 0; i < kSVec4; ++i) {
                const bool on = (pass >> i) & 1u;
                const uint32_t bl = __ballot_sync(0xffffffffu, on);
                if (on) list[total + __popc(bl & lt)] = static_cast<uint16_t>(i * kSThreads + tid);
                total += __popc(bl);
            }
            __syncwarp();
            const SeedRec sr{r.B, r.cB, r.bcol, 0};
            for (int m = lane; m < total; m += 32) {
                const int f = list[m];
                const float4 x4 = piece[f];
                const int c4 = col0 + 4 * f;
                const uint4 nw = noise_group(p.rk[0], grow, static_cast<uint32_t>(c4 >> 2));
                const uint32_t wmax = max(max(nw.x, nw.y), max(nw.z, nw.w));
                const float mx = max4f(x4);
                const float emax = RAW ? ex2_ftz(fmaf(mx, r.ls, -r.cB))
                                       : ex2_ftz(fmaf(sq.exact(mx) - r.B, kLog2e, kRaceSlack));
                if (one_minus_u_lower(wmax) <= emax) {
                    const float4 e = race_e(x4, RAW, r.ls, sr, sq);
                    uint32_t bits = 0;
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (one_minus_u_lower(word_of(nw, q)) <= comp(e, q)) bits |= 1u << q;
                    if (bits) {
                        const Best b2 = race_rescore(bits, x4, nw, c4, r.bcol, sq, Best{lb.wb, lb.wc});
                        lb.wb = b2.s;
                        lb.wc = b2.c;
                    }
                }
            }
            __syncwarp();  // the list is rewritten for the next piece
        }
    }

    // top-k candidates x >= thr (rare: the slots reaching it)
    if ((r.flags & kFTopk) && mthr >= r.thr) {
        uint32_t km = 0;
#pragma unroll
        for (int i = 0; i < kSVec4; ++i) km |= (m4[i] >= r.thr ? 1u : 0u) << i;
        if (km) topk_collect(km, piece, tid, col0, ncols, r.thr, sq, &sh.tile_nk, p.keys + t * kTileKeys);
    }
}

template <int PD>
__device__ __forceinline__ void phase_b_any(const SplitParams& p, ClusterSmem& sh, const CRow& r,
                                            const ScaledQuotient& sq, const float4* piece, uint64_t grow,
                                            int64_t row, int col0, int ncols, int64_t t, bool stats, int tid,
                                            int lane, int warp, LaneBest& lb) {
    if (r.flags & kFRaw)
        phase_b<PD, true>(p, sh, r, sq, piece, grow, row, col0, ncols, t, stats, tid, lane, warp, lb);
    else
        phase_b<PD, false>(p, sh, r, sq, piece, grow, row, col0, ncols, t, stats, tid, lane, warp, lb);
}

// ------------------------------------------------------ the kernel

// Grid: clusters of C CTAs (C = the cluster size of the launch); cluster q
// takes list entries li_begin + q, + nclusters, ... Every CTA owns columns
// [rank * chunk_cols, min(V, (rank + 1) * chunk_cols)) of each of its rows.
template <int PD>
__global__ void __launch_bounds__(kSThreads, 3) split_cluster(const __grid_constant__ SplitParams p,
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
    const int P = cs.pieces;
    const bool stats = p.stats != 0;
    const int lend = list_end(p);

    // the buffer past this CTA's columns reads as -inf (never copied into)
    for (int f = (ncols >> 2) + tid; f < P * kCPieceF4; f += kSThreads)
        buf[f] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    if (tid == 0) {
        for (int j = 0; j < kCMaxPieces; ++j) {
            mbar_init(&sh.piece_full[j], 1);
            sh.piece_count[j] = 0;
            sh.last_issue[j] = -1;
        }
        mbar_init(&sh.part_full[0], 1);
        mbar_init(&sh.part_full[1], 1);
        sh.abort = 0;
        sh.tile_nk = 0;
        fence_barrier_init();
        // rows 0 and 1 of the cluster: C parts of 96 bytes each
        mbar_arrive_expect_tx(&sh.part_full[0], kCPartWords * 16u * C);
        mbar_arrive_expect_tx(&sh.part_full[1], kCPartWords * 16u * C);
    }
    __syncthreads();
    cluster_sync_all();  // every CTA's barriers are set before any push

    int li = p.li_begin + static_cast<int>(cluster_index());
    if (tid == 0 && li < lend)
        for (int j = 0; j < P; ++j) issue_piece(p, sh, buf, j, li, 0, c0, ncols);

    for (int it = 0; li < lend; ++it, li += ncl) {
        const int64_t row = p.list1[li];
        const RowTemp rt = p.rt[row];
        const ScaledQuotient sq{rt.qt, rt.qy, rt.qmode};
        const uint64_t grow = static_cast<uint64_t>(p.row0 + row);
        const bool kept = p.map_row || p.keep == nullptr || p.keep[slot_of(p, grow)] != 0;
        const bool topk = p.k > 0 && kept;
        const bool noisy = stats && rt.temp > 0.0f;
        const int s = it & 1;

        // ---- phase A
        for (int j = 0; j < P; ++j) {
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(&sh.piece_full[j], static_cast<uint32_t>(it & 1)))) {
                if (lane == 0) {
                    sh.abort = 1;
                    raise_device_error(p.err, 1);
                }
                break;
            }
            const WarpPart wp = phase_a(buf + j * kCPieceF4, sq, c0 + j * kCPieceCols, tid, stats);
            if (lane == 0) sh.wparts[j][warp] = wp;
        }
        __syncthreads();
        if (sh.abort) break;

        // ---- the CTA's part to every CTA; the merge of the C parts
        if (warp == 0) {
            make_part(p, sh, sq, grow, noisy, P, ncols, c0, cs.top_m, s, rank, C, lane);
            const bool ok = __all_sync(
                0xffffffffu, mbar_wait_cluster_bounded(&sh.part_full[s], static_cast<uint32_t>((it >> 1) & 1)));
            if (!ok) {
                if (lane == 0) {
                    sh.abort = 1;
                    raise_device_error(p.err, 1);
                }
            } else {
                if (static_cast<int>(C) * cs.top_m <= 64)
                    merge_parts<2>(p, sh, rt, row, stats, topk, cs.top_m, s, rank, C, lane);
                else
                    merge_parts<8>(p, sh, rt, row, stats, topk, cs.top_m, s, rank, C, lane);
                __syncwarp();
                // the slot takes the parts of row it + 2
                if (lane == 0) mbar_arrive_expect_tx(&sh.part_full[s], kCPartWords * 16u * C);
            }
        }
        __syncthreads();
        if (sh.abort) break;

        // ---- phase B
        const CRow r = sh.row;
        const int64_t t = static_cast<int64_t>(li) * C + rank;  // the CTA's tile record
        const int li_next = li + ncl;
        const bool has_next = li_next < lend;
        LaneBest lb{r.B, r.bcol, INT_MAX};
        for (int j = 0; j < P; ++j) {
            phase_b_any<PD>(p, sh, r, sq, buf + j * kCPieceF4, grow, row, c0 + j * kCPieceCols,
                            piece_cols(ncols, j), t, stats, tid, lane, warp, lb);
            // the last warp out of the piece starts the next row's copy into it
            if (release_stage(&sh.piece_count[j], lane) && has_next && lane == 0) {
                fence_proxy_async_smem();
                issue_piece(p, sh, buf, j, li_next, it + 1, c0, ncols);
            }
        }
        warp_best(lb.wb, lb.wc);
        lb.acand = warp_min_nonneg(lb.acand);
        if (lane == 0) {
            sh.best_s[warp] = lb.wb;
            sh.best_c[warp] = lb.wc;
            sh.best_a[warp] = lb.acand;
        }
        __syncthreads();
        if (warp == 0) {
            float b = lane < kSWarps ? sh.best_s[lane] : -INFINITY;
            int bc = lane < kSWarps ? sh.best_c[lane] : INT_MAX;
            warp_best(b, bc);
            const int a = warp_min_nonneg(lane < kSWarps ? sh.best_a[lane] : INT_MAX);
            if (lane == 0) {
                p.tb[t] = TileSeed{b, bc};
                p.te[t] = TileEnd{(r.flags & kFTopk) ? sh.tile_nk : 0, a};
                sh.tile_nk = 0;
            }
        }
    }
    asm volatile("griddepcontrol.launch_dependents;");
    if (sh.abort && tid == 0) {
        // copies still in flight land before the shared memory is released
        for (int j = 0; j < P; ++j)
            if (sh.last_issue[j] >= 0)
                mbar_wait_bounded(&sh.piece_full[j], static_cast<uint32_t>(sh.last_issue[j] & 1));
    }
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
    cs.pieces = (chunk + kCPieceCols - 1) / kCPieceCols;
    // each CTA publishes its largest group maxima: enough that about 2k of
    // them reach the merge (the threshold's quality)
    const int groups = cs.pieces * kSWarps;
    const int m = k > 0 ? (2 * k + C - 1) / C : 1;
    cs.top_m = m > groups ? groups : m;
    *out = cs;
    *cluster_size = C;
    return true;
}

drs_status cluster_launch(const SplitParams& p, const ClusterShape& cs, int C, int64_t rows,
                          cudaStream_t stream) {
    const size_t smem = static_cast<size_t>(cs.pieces) * kCPieceCols * 4;
    void (*kernel)(SplitParams, ClusterShape) =
        p.probs_dtype == 1 ? split_cluster<1> : p.probs_dtype == 2 ? split_cluster<2> : split_cluster<0>;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
            cudaSuccess ||
        cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
        return DRS_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kSThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(C);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    // as many clusters as can be resident at once (each loops over rows),
    // no more than rows
    cfg.gridDim = dim3(static_cast<unsigned>(C));
    int active = 0;
    if (cudaOccupancyMaxActiveClusters(&active, kernel, &cfg) != cudaSuccess || active < 1) return DRS_ERR_CUDA;
    const int64_t ncl = rows < active ? rows : active;
    cfg.gridDim = dim3(static_cast<unsigned>(ncl * C));
    return cudaLaunchKernelEx(&cfg, kernel, p, cs) == cudaSuccess ? DRS_OK : DRS_ERR_CUDA;
}

}  // namespace rs
}  // namespace drs
