// row_common.cuh -- definitions shared by the two implementations of the row
// statistics (row_split.cu: two streaming passes; row_cluster.cu: one read
// per row by a thread-block cluster): tile geometry, the per-row and
// per-tile records, the launch parameters, and device helpers (order keys,
// top-k keys, rounding to bf16/fp16, the Philox noise of a group of four
// columns, the exact rescoring of Gumbel-race survivors, top-k candidate
// collection).
#pragma once

#include <cfloat>
#include <climits>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "drs_device.cuh"
#include "drs_internal.h"

namespace drs {
namespace rs {

constexpr int kSThreads = 256;
constexpr int kSWarps = kSThreads / 32;
#ifndef DRS_SPLIT_VEC4
#define DRS_SPLIT_VEC4 8
#endif
#ifndef DRS_SPLIT_STAGES
#define DRS_SPLIT_STAGES 2
#endif
#ifndef DRS_P1_MINB
#define DRS_P1_MINB 3
#endif
#ifndef DRS_P2_MINB
#define DRS_P2_MINB 3
#endif
#ifndef DRS_P1_VEC4
#define DRS_P1_VEC4 6
#endif
constexpr int kSVec4 = DRS_SPLIT_VEC4;             // pass 2: float4 slots per thread
constexpr int kTileCols = kSThreads * kSVec4 * 4;  // 8192 columns per pass-2 tile
constexpr int kMaxTiles = (DRS_MAX_VOCAB + kTileCols - 1) / kTileCols;
// Pass 1 has tiles of its own (measured: it streams faster with 24 KiB tiles
// than with pass 2's 32 KiB ones, pass 2 the other way round).
constexpr int kP1Vec4 = DRS_P1_VEC4;
constexpr int kP1Cols = kSThreads * kP1Vec4 * 4;   // 6144 columns per pass-1 tile
constexpr int kMaxTiles1 = (DRS_MAX_VOCAB + kP1Cols - 1) / kP1Cols;
// warp maxima per thread in the merge: rows of up to 60 pass-1 tiles
// (368640 columns) take one warp; longer rows, up to the longest, share the
// kWideMergeWarps warps of a CTA
constexpr int kOrdSmall = (60 * kSWarps + 31) / 32;
constexpr int kWideMergeWarps = 8;
constexpr int kOrdWide = (kMaxTiles1 * kSWarps + 32 * kWideMergeWarps - 1) / (32 * kWideMergeWarps);
constexpr int kTilesSmall = (60 + 31) / 32;  // tiles per lane in the finish
constexpr int kTilesLarge = (kMaxTiles + 31) / 32;
constexpr int kStages = DRS_SPLIT_STAGES;          // tiles in flight per CTA
constexpr int kStageF4 = kTileCols / 4;             // float4 per stage
constexpr size_t kStageBytes = kTileCols * 4;       // 32 KiB
constexpr int kMap = 64;                            // tile -> row map, a ring
constexpr int kTileKeys = 32;     // top-k candidates a tile keeps
constexpr int kRowKeys = 512;     // top-k candidates a row merges
constexpr int kSplitMaxK = 64;    // larger k: the exact kernel
constexpr int kHardOffset = 64;   // hard-row list: count at [0], rows from [64]
constexpr int kCount1 = 1;        // header word: length of the row list
constexpr int kMaxSeeds = 8;      // noise seeds of one call
constexpr float kRawLimit = 256.0f;
// Slack (log2 units) of the race bounds: covers the roundings of the
// reference c and of x * log2(e) / Te (a few 1e-5 for |s| up to a few
// hundred).
constexpr float kRaceSlack = 0x1p-10f;

// A pass-1 row: its temperature and the quotient constants (16 bytes).
struct alignas(16) RowTemp {
    float temp;
    float qt;
    float qy;
    int qmode;
};

// Pass-1 record of a tile (96 bytes).
struct alignas(16) TileStats {
    float m;      // max exact quotient (-inf: none)
    float s;      // sum e^(s - m)
    float w;      // sum e^(s - m) (s - m)
    int arg;      // lowest column holding the raw max (the tile's first column if none)
    float xmax;   // raw max
    int pad[3];
    uint32_t wmax[kSWarps];  // order keys of the warps' raw maxima, 0: no columns
    int wcol[kSWarps];       // lowest column holding each warp's raw max (INT_MAX: none)
};
static_assert(sizeof(TileStats) == 96, "tile record");

enum : int { kFNoisy = 1, kFTopk = 2, kFRaw = 4 };

// A row after the merge (64 bytes), followed in the row's entry by one
// SeedRec per noise seed.
struct alignas(16) RowRecord {
    float M;      // max scaled logit (exact), -inf: the row is -inf everywhere
    float log2s;  // log2 S
    float ls;     // RN(log2(e) * RN(1/Te))
    float c2;     // raw rows: RN(RN(Mraw * ls) + log2 S)
    float thr;    // top-k threshold (raw logit)
    float lns;    // log S
    int arg;      // lowest column holding the raw row max
    int flags;
    float qt, qy;
    int qmode;
    float cthr;   // a logit whose exact quotient equals M is at least this
    int pad[4];
};
static_assert(sizeof(RowRecord) == 64, "row record");

// The race bound of one seed for a row (16 bytes).
struct alignas(16) SeedRec {
    float B;      // best Gumbel-max score among the warps' candidates
    float cB;     // raw rows: RN(RN(Mraw * ls) + (B - M) log2(e)) - slack
    int bcol;     // its column
    int pad;
};
constexpr size_t kRowEntryMax = sizeof(RowRecord) + kMaxSeeds * sizeof(SeedRec);

// Pass-2 record of a tile: candidate count and the lowest column below the
// raw max whose exact quotient is M (8 bytes); per seed, the race winner.
struct alignas(8) TileEnd {
    int nk;
    int acol;
};
struct alignas(8) TileSeed {
    float b;
    int col;
};

struct SplitParams {
    const float* logits;
    int64_t row_stride;
    int64_t rows;
    int64_t row0;
    int64_t canvas_len;
    const float* temps;
    const uint8_t* keep;
    int64_t* argmax;
    int64_t* sample;      // [n_seeds, rows]
    float* entropy;
    void* probs;
    int64_t probs_row_stride;
    int32_t* out_ids;
    float* out_lp;
    int32_t* hard;    // header (hard count, list lengths), then hard rows
    int32_t* list1;   // the rows the passes work on
    RowTemp* rt;
    TileStats* ts;    // by tile (list index * G + tile of the row)
    unsigned char* rr;  // by row: RowRecord + n_seeds SeedRec (rec_bytes each)
    TileEnd* te;      // by tile
    TileSeed* tb;     // by tile and seed
    uint64_t* keys;   // by tile
    // Row map (the stash): rows are entries e < *map_count of a list, read
    // from logits row map_row[e] with temperature map_temp[e], all kept;
    // null for the ordinary calls. out_m / out_logs (or null) receive each
    // row's max scaled logit and log S from the merge.
    const int32_t* map_row;
    const float* map_temp;
    const int32_t* map_count;
    float* out_m;
    float* out_logs;
    // The list entries of this launch: the whole list (li_part 0), or with
    // the list of n entries divided at h = floor(n * li_num / li_den) (n is
    // known on the device only), its head [0, h) (1) or its tail [h, n) (2).
    int li_part;
    int li_num;
    int li_den;
    int* err;
    PhiloxRoundKeys rk[kMaxSeeds];
    int n_seeds;
    int rec_bytes;    // sizeof(RowRecord) + n_seeds * sizeof(SeedRec)
    int vocab;
    int tiles_per_row;  // pass-2 tiles of a row (the finish's records)
    int tiles1;         // pass-1 tiles of a row (the merge's records)
    int vec;          // rows start 16-byte aligned: bulk copies
    int probs_dtype;  // 0 none, 1 bf16, 2 fp16
    int probs_vec;    // 8-byte probability stores
    int index32;
    int stats;
    int k;
    int fault;        // test hook: CTA 0 withholds its first tile of pass 1
};

// ------------------------------------------------------------ helpers

__device__ __forceinline__ uint64_t slot_of(const SplitParams& p, uint64_t grow) {
    return p.index32 ? static_cast<uint64_t>(static_cast<uint32_t>(grow) /
                                             static_cast<uint32_t>(p.canvas_len))
                     : grow / static_cast<uint64_t>(p.canvas_len);
}

__device__ __forceinline__ void set_comp(float4& v, int q, float x) {
    if (q == 0) v.x = x;
    else if (q == 1) v.y = x;
    else if (q == 2) v.z = x;
    else v.w = x;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ float max4f(const float4& v) { return max3(v.x, v.y, fmaxf(v.z, v.w)); }

__device__ __forceinline__ float min3(float a, float b, float c) {
    float r;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// 2^x with subnormal results flushed to zero (a single special-function
// instruction).
__device__ __forceinline__ float ex2_ftz(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Order-preserving unsigned form of an fp32 value (-inf lowest, above 0).
__device__ __forceinline__ uint32_t ord32(float x) {
    const uint32_t b = __float_as_uint(x);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float unord32(uint32_t o) {
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}
constexpr uint32_t kOrdNegInf = 0x007FFFFFu;

// Top-k key: the value (-0.0 as +0.0) in the high word, then the lower
// column first (the _lp_topk_kernel key order).
__device__ __forceinline__ uint64_t topk_key(float s, int col) {
    return (static_cast<uint64_t>(ord32(s + 0.0f)) << 32) |
           static_cast<uint32_t>(0x7FFFFFFF - col);
}
__device__ __forceinline__ float key_value(uint64_t key) {
    return unord32(static_cast<uint32_t>(key >> 32));
}
__device__ __forceinline__ int key_col(uint64_t key) {
    return 0x7FFFFFFF - static_cast<int>(static_cast<uint32_t>(key));
}

// Two values rounded to nearest even and packed (a in the low half), in one
// conversion instruction.
template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
    uint32_t r;
    if (BF16) asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
    else asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
    return r;
}

// Philox4x32-10 of (group, 0, row) with the per-seed round keys: each round's
// two 32x32->64 products taken as one wide multiplication each.
__device__ __forceinline__ uint4 noise_group(const PhiloxRoundKeys& rk, uint64_t row,
                                             uint32_t group) {
    uint32_t c0 = group, c1 = 0u, c2 = static_cast<uint32_t>(row), c3 = static_cast<uint32_t>(row >> 32);
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        uint64_t pa, pb;
        asm("mul.wide.u32 %0, %1, %2;" : "=l"(pa) : "r"(c0), "r"(0xD2511F53u));
        asm("mul.wide.u32 %0, %1, %2;" : "=l"(pb) : "r"(c2), "r"(0xCD9E8D57u));
        const uint32_t hi_a = static_cast<uint32_t>(pa >> 32), lo_a = static_cast<uint32_t>(pa);
        const uint32_t hi_b = static_cast<uint32_t>(pb >> 32), lo_b = static_cast<uint32_t>(pb);
        c0 = hi_b ^ c1 ^ rk.k0[r];
        c1 = lo_b;
        c2 = hi_a ^ c3 ^ rk.k1[r];
        c3 = lo_a;
    }
    return make_uint4(c0, c1, c2, c3);
}

// The same Philox4x32-10 of (group, 0, row) with the first two rounds folded
// per row: round 1 multiplies the row's low word, which is the same for
// every group of the row, and round 2 multiplies round 1's first output word,
// which then is too. Per group that leaves one multiplication in each of the
// first two rounds (18 wide multiplications instead of 20).
struct RowNoise {
    uint32_t c1;    // round 1: low half of MB * lo32(row)
    uint32_t x3;    // hi32(row) ^ k1[0]
    uint32_t y0;    // round 2: c1 ^ k0[1]
    uint32_t y2;    // round 2: high half of MA * c0 ^ k1[1]
    uint32_t c3;    // round 2: low half of MA * c0
};

__device__ __forceinline__ RowNoise row_noise(const PhiloxRoundKeys& rk, uint64_t row) {
    uint64_t pb, pa;
    asm("mul.wide.u32 %0, %1, %2;" : "=l"(pb) : "r"(static_cast<uint32_t>(row)), "r"(0xCD9E8D57u));
    const uint32_t c0 = static_cast<uint32_t>(pb >> 32) ^ rk.k0[0];  // round 1's first word
    RowNoise rn;
    rn.c1 = static_cast<uint32_t>(pb);
    rn.x3 = static_cast<uint32_t>(row >> 32) ^ rk.k1[0];
    asm("mul.wide.u32 %0, %1, %2;" : "=l"(pa) : "r"(c0), "r"(0xD2511F53u));
    rn.y0 = rn.c1 ^ rk.k0[1];
    rn.y2 = static_cast<uint32_t>(pa >> 32) ^ rk.k1[1];
    rn.c3 = static_cast<uint32_t>(pa);
    return rn;
}

__device__ __forceinline__ uint4 noise_folded(const PhiloxRoundKeys& rk, const RowNoise& rn, uint32_t group) {
    uint64_t pa, pb;
    // round 1: (group, 0, lo, hi) -> (c0, c1, hi(MA g) ^ x3, lo(MA g))
    asm("mul.wide.u32 %0, %1, %2;" : "=l"(pa) : "r"(group), "r"(0xD2511F53u));
    const uint32_t r1c2 = static_cast<uint32_t>(pa >> 32) ^ rn.x3;
    const uint32_t r1c3 = static_cast<uint32_t>(pa);
    // round 2: (c0, c1, r1c2, r1c3) -> (hi(MB r1c2) ^ c1 ^ k0, lo(MB r1c2), hi(MA c0) ^ r1c3 ^ k1, lo(MA c0))
    asm("mul.wide.u32 %0, %1, %2;" : "=l"(pb) : "r"(r1c2), "r"(0xCD9E8D57u));
    uint32_t c0 = static_cast<uint32_t>(pb >> 32) ^ rn.y0;
    uint32_t c1 = static_cast<uint32_t>(pb);
    uint32_t c2 = rn.y2 ^ r1c3;
    uint32_t c3 = rn.c3;
#pragma unroll
    for (int r = 2; r < 10; ++r) {
        asm("mul.wide.u32 %0, %1, %2;" : "=l"(pa) : "r"(c0), "r"(0xD2511F53u));
        asm("mul.wide.u32 %0, %1, %2;" : "=l"(pb) : "r"(c2), "r"(0xCD9E8D57u));
        const uint32_t hi_a = static_cast<uint32_t>(pa >> 32), lo_a = static_cast<uint32_t>(pa);
        const uint32_t hi_b = static_cast<uint32_t>(pb >> 32), lo_b = static_cast<uint32_t>(pb);
        c0 = hi_b ^ c1 ^ rk.k0[r];
        c1 = lo_b;
        c2 = hi_a ^ c3 ^ rk.k1[r];
        c3 = lo_a;
    }
    return make_uint4(c0, c1, c2, c3);
}

// Rows whose scaled values are too large for the raw domain take exact
// quotients s = x / Te, with exponentials 2^((s - m) log2 e) against a
// reference m = the exact quotient of a raw max xm. A logit far enough
// below xm gives an exponential that is exactly 0 after flushing (for
// bf16 probabilities too, whose exponent is lifted by 64), however the
// quotients round, so its quotient need not be taken. The test is raw:
// t = x yl - xm yl by one fused multiply-add, yl = RN(log2(e) RN(1/Te)),
// against a limit that covers the roundings of 1/Te, of both quotients, of
// their difference and of t itself (each within 2^-21 of |x yl| + |xm yl|):
// t < -257 - 2^-19 |xm yl| implies (s - m) log2(e) < -256. A -inf logit
// passes it (t = -inf). Used only for reading: a logit that passes is
// given a large finite stand-in, never -inf, so that e t stays 0.
struct FarBelow {
    float yl, c, lim;
    __device__ __forceinline__ FarBelow(float xm, float yl_) : yl(yl_) {
        c = xm * yl_;
        lim = -257.0f - fabsf(c) * 0x1p-19f;
    }
    __device__ __forceinline__ bool operator()(float x) const { return fmaf(x, yl, -c) < lim; }
};
constexpr float kFarStandIn = -1e30f;  // exponent far below any exponential's range

// The list entries of this launch: [list_begin, list_end).
__device__ __forceinline__ int list_split(const SplitParams& p, int n) {
    return static_cast<int>(static_cast<int64_t>(n) * p.li_num / p.li_den);
}
__device__ __forceinline__ int list_begin(const SplitParams& p) {
    return p.li_part == 2 ? list_split(p, p.hard[kCount1]) : 0;
}
__device__ __forceinline__ int list_end(const SplitParams& p) {
    const int n = p.hard[kCount1];
    return p.li_part == 1 ? list_split(p, n) : n;
}

// A warp's part of a tile's statistics: the raw max and its lowest column,
// S and W relative to the reference of the warp.
struct WarpPart {
    float m, s, w, xmax;
    int arg;
};

// e^(s - B) of a group, over-estimated by the slack: 2^(x ls - cB) on raw
// rows, else from the exact quotients (flushed below 2^-126: such elements
// cannot win).
__device__ __forceinline__ float4 race_e(const float4& x, bool raw, float ls, const SeedRec& sr,
                                         const ScaledQuotient& sq) {
    float4 e;
    if (raw) {
        e.x = ex2_ftz(fmaf(x.x, ls, -sr.cB));
        e.y = ex2_ftz(fmaf(x.y, ls, -sr.cB));
        e.z = ex2_ftz(fmaf(x.z, ls, -sr.cB));
        e.w = ex2_ftz(fmaf(x.w, ls, -sr.cB));
    } else {
        e.x = ex2_ftz(fmaf(sq.exact(x.x) - sr.B, kLog2e, kRaceSlack));
        e.y = ex2_ftz(fmaf(sq.exact(x.y) - sr.B, kLog2e, kRaceSlack));
        e.z = ex2_ftz(fmaf(sq.exact(x.z) - sr.B, kLog2e, kRaceSlack));
        e.w = ex2_ftz(fmaf(sq.exact(x.w) - sr.B, kLog2e, kRaceSlack));
    }
    return e;
}

struct Best {
    float s;
    int c;
};

// The survivors `bits` of the group at column c4 scored exactly (s + g)
// against the best so far; the column of B was scored already.
static __device__ __noinline__ Best race_rescore(uint32_t bits, const float4 x4, uint4 nw, int c4,
                                          int bcol, ScaledQuotient sq, Best best) {
    while (bits) {
        const int q = __ffs(bits) - 1;
        bits &= bits - 1;
        const int col = c4 + q;
        if (col == bcol) continue;
        const float score = sq.exact(comp(x4, q)) + gumbel_of_bits(word_of(nw, q));
        if (beats(score, col, best.s, best.c)) best = Best{score, col};
    }
    return best;
}

// The top-k candidates of a thread's slots in `smask` (slot i: bit i): the
// logits x >= thr, read again from the stage, keyed by (exact value, lower
// column) into the tile's list.
static __device__ __noinline__ void topk_collect(uint32_t smask, const float4* stage, int tid, int col0,
                                          int ncols, float thr, ScaledQuotient sq, int* count,
                                          uint64_t* kdst) {
    while (smask) {
        const int f = (__ffs(smask) - 1) * kSThreads + tid;
        smask &= smask - 1;
        const float4 x4 = stage[f];
        for (int q = 0; q < 4; ++q) {
            const float x = comp(x4, q);
            if (4 * f + q < ncols && x >= thr) {
                const int pos = atomicAdd(count, 1);
                if (pos < kTileKeys) kdst[pos] = topk_key(sq.exact(x), col0 + 4 * f + q);
            }
        }
    }
}

// Count a warp out of a stage; true on the warp that counted out last (the
// count is reset for the stage's next tile).
__device__ __forceinline__ bool release_stage(int* count, int lane) {
    int last = 0;
    __syncwarp();
    if (lane == 0) {
        __threadfence_block();
        last = atomicAdd(count, 1) == kSWarps - 1;
        if (last) *count = 0;
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (last) __threadfence_block();
    return last != 0;
}

// The one-read path (row_cluster.cu): a row split over the CTAs of a
// thread-block cluster, the CTAs' partial results merged through distributed
// shared memory. ClusterShape: columns per CTA (a multiple of 4), pieces of
// 8192 columns per CTA, and how many of its largest group maxima each CTA
// contributes to the row's top-k threshold.
struct ClusterShape {
    int chunk_cols;
    int pieces;
    int top_m;
};
// Whether the cluster path takes a call (rows start 16-byte aligned, vocab a
// multiple of 4 and at most 262144, one seed, k <= 64); its shape and cluster
// size.
bool cluster_plan(int64_t rows, int64_t vocab, int32_t k, int32_t n_seeds, bool aligned16, ClusterShape* out,
                  int* cluster_size);
// How a call's rows are shared (see split_plan_query in drs_internal.h): the
// last `tail` rows of the list go to the two passes on the free SMs.
struct RowSplitPlan {
    ClusterShape shape;
    int cluster_size;
    int clusters;
    int free_sms;
    int head_num, head_den;  // the head's share of the row list
    int64_t tail;            // the tail of a list of `rows` entries
};
bool row_split_plan(int64_t rows, int64_t vocab, int32_t k, int32_t n_seeds, bool aligned16, int probs_dtype,
                    bool stats, RowSplitPlan* out);

// Clusters of the cluster kernel resident at once on the current device
// (0 on failure).
int cluster_active(int probs_dtype, int cluster_size);
// Launch the cluster kernel on the list entries of p (after
// split_prep, before split_finish; the CTA of rank r writes tile r of its
// row's tiles_per_row records, tile r + cluster_size empty when it exists).
drs_status cluster_launch(const SplitParams& p, const ClusterShape& cs, int cluster_size, int64_t rows,
                          cudaStream_t stream);

}  // namespace rs
}  // namespace drs
