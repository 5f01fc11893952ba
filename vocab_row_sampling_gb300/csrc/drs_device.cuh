// drs_device.cuh -- device building blocks shared by the libdrs kernels:
// the Philox4x32-10 noise generator and the Gumbel noise of a word, bounded
// mbarrier waits, the bulk-copy (TMA) loads that stage data in shared
// memory, warp reductions, the exact temperature quotient, and the team
// plan of the exact top-k kernel (CTAs that share one row).
#pragma once

#include <climits>
#include <cstdint>
#include <cuda_runtime.h>

namespace drs {

constexpr int kThreads = 512;               // threads per CTA of the exact top-k kernel
constexpr int kWarps = kThreads / 32;
constexpr size_t kSmemPerSm = 233472;       // shared memory of one SM (228 KB)
constexpr size_t kSmemPerCta = 232448;      // largest opt-in per CTA (227 KB)
constexpr size_t kSmemReserved = 1024;      // the driver's share of each CTA
constexpr int kMaxTeam = 32;                // CTAs that share one row (one per lane of the merging warp)
constexpr int kRing = 8;                    // exchange slots per CTA
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kTempFloor = 1e-10f;        // clamp(min=1e-10) of the temperature

// Bounded waits: a wait that has not completed after this many nanoseconds
// gives up, raises the device error flag and makes its kernel skip the rest
// of its work.
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------- Philox

// Philox4x32-10, the counter-based generator of Salmon, Moraes, Dror and
// Shaw (SC'11): ten rounds of two 32x32->64 multiplications whose high
// halves are mixed with the other two words and the round key, the key
// advancing by a Weyl sequence between rounds.
struct PhiloxKey {
    uint32_t k0, k1;
};

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, PhiloxKey key) {
    constexpr uint32_t kMulA = 0xD2511F53u, kMulB = 0xCD9E8D57u;
    constexpr uint32_t kWeylA = 0x9E3779B9u, kWeylB = 0xBB67AE85u;
    uint32_t k0 = key.k0, k1 = key.k1;
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint32_t hi_a = __umulhi(kMulA, c.x);
        const uint32_t lo_a = kMulA * c.x;
        const uint32_t hi_b = __umulhi(kMulB, c.z);
        const uint32_t lo_b = kMulB * c.z;
        c = make_uint4(hi_b ^ c.y ^ k0, lo_b, hi_a ^ c.w ^ k1, lo_a);
        k0 += kWeylA;
        k1 += kWeylB;
    }
    return c;
}

// The ten round keys of one seed, computed once on the host: a kernel that
// reads them from its parameters saves the key schedule per call.
struct PhiloxRoundKeys {
    uint32_t k0[10];
    uint32_t k1[10];

    static PhiloxRoundKeys of(uint64_t seed) {
        PhiloxRoundKeys rk;
        uint32_t a = static_cast<uint32_t>(seed), b = static_cast<uint32_t>(seed >> 32);
        for (int r = 0; r < 10; ++r) {
            rk.k0[r] = a;
            rk.k1[r] = b;
            a += 0x9E3779B9u;
            b += 0xBB67AE85u;
        }
        return rk;
    }
};

// The four noise words of columns 4*group .. 4*group+3 of `row`.
__device__ __forceinline__ uint4 noise_words(PhiloxKey key, uint64_t row,
                                             uint64_t group) {
    return philox4x32_10(make_uint4(static_cast<uint32_t>(group),
                                    static_cast<uint32_t>(group >> 32),
                                    static_cast<uint32_t>(row),
                                    static_cast<uint32_t>(row >> 32)),
                         key);
}

__device__ __forceinline__ uint32_t word_of(uint4 w, int q) {
    return q == 0 ? w.x : q == 1 ? w.y : q == 2 ? w.z : w.w;
}

// Exponential variate E = -log(u), u = max((bits >> 8) * 2^-24, 1e-20f).
// For u >= 1/2 the logarithm is taken as log1p(-(1 - u)) with 1 - u exact,
// so E keeps its relative accuracy when u is close to 1.
__device__ __forceinline__ float exponential_of_bits(uint32_t bits) {
    const uint32_t n = bits >> 8;
    if (n < (1u << 23)) {
        const float u = fmaxf(static_cast<float>(n) * 0x1p-24f, 1e-20f);
        return -logf(u);
    }
    const float one_minus_u = static_cast<float>((1u << 24) - n) * 0x1p-24f;
    return -log1pf(-one_minus_u);
}

// The Gumbel noise -log(-log u) of one noise word, fp32.
__device__ __forceinline__ float gumbel_of_bits(uint32_t bits) {
    return -logf(exponential_of_bits(bits));
}

// A lower bound of 1 - u, itself a lower bound of E = -log(u), from the
// top 23 bits of the word without an int-to-float conversion: with
// u' = 1 + (bits >> 9) * 2^-23 in [1, 2), u <= u' - 1 + 2^-24, so
// 1 - u >= (2 - 2^-24) - u'.
__device__ __forceinline__ float one_minus_u_lower(uint32_t bits) {
    return 0x1.fffffep0f - __uint_as_float(0x3F800000u | (bits >> 9));
}


// ------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// A plain arrival (release at CTA scope): no transaction bytes.
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// try_wait that lets the hardware suspend the thread until the phase
// completes or `hint_ns` pass, so that a waiting warp issues nothing.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint64_t* bar, uint32_t parity,
                                                      uint32_t hint_ns) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return done != 0;
}

// Wait for the phase with the given parity to complete; false if it has not
// completed within kWaitLimitNs. Each try suspends the thread for up to
// 100 us rather than spinning.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait_suspend(bar, parity, 100000u)) return true;
        if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// Bulk global -> shared copy (the non-tensor TMA path). dst and src must be
// 16-byte aligned and bytes a multiple of 16. Completion is signalled on
// `bar` as transaction bytes. evict_first: the logits are read once.
__device__ __forceinline__ void tma_load_1d(void* dst, const void* src, uint32_t bytes,
                                            uint64_t* bar) {
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// --------------------------------------------------------- reductions

__device__ __forceinline__ float warp_max(float v) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

// Best (score, column): larger score wins, equal scores go to the lower
// column. Columns of "no candidate" are INT32_MAX with score -inf.
__device__ __forceinline__ bool beats(float s, int c, float bs, int bc) {
    return s > bs || (s == bs && c < bc);
}

// Warp-wide reductions in one instruction each (redux.sync): max of floats
// (NaN inputs ignored), min of non-negative ints.
__device__ __forceinline__ float warp_max_f(float v) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

__device__ __forceinline__ int warp_min_nonneg(int v) {
    uint32_t r;
    asm volatile("redux.sync.min.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(static_cast<uint32_t>(v)));
    return static_cast<int>(r);
}

// The best (score, column) of the warp, on every lane: the largest score,
// then the lowest column among the lanes holding it. Scores are finite or
// -inf (never NaN).
__device__ __forceinline__ void warp_best(float& s, int& c) {
    const float top = warp_max_f(s);
    c = warp_min_nonneg(s == top ? c : INT_MAX);
    s = top;
}

__device__ __forceinline__ void raise_device_error(int* flag, int code) {
    if (flag) atomicExch(flag, code);
}

// ------------------------------------------------------ work planning

// How rows are split over CTAs: `team` CTAs share a row, each owning
// `chunk` columns (a multiple of 4); `num_teams` teams take rows round
// robin; `vec4` float4 slots per thread cover a chunk; `ctas_per_sm` CTAs
// are resident per SM.
struct RowPlan {
    int team;
    int chunk;
    int num_teams;
    int vec4;
    int ctas_per_sm;
};

inline size_t smem_per_cta(int ctas_per_sm) {
    return ctas_per_sm >= 2 ? kSmemPerSm / ctas_per_sm - kSmemReserved : kSmemPerCta;
}

// Choose the team size G that minimises the per-CTA work
// ceil(rows / teams) * chunk, with teams = min(rows, capacity / G); ties go
// to the smaller G (fewer records to merge). With two_per_sm, rows up to
// kMaxTeam * 8192 columns use 16 logits per thread and two CTAs per SM;
// longer rows (and two_per_sm == false) use up to 32 logits per thread and
// one CTA per SM.
inline RowPlan plan_rows(int64_t rows, int vocab, int sms, bool two_per_sm = true) {
    const bool pair = two_per_sm && vocab <= kMaxTeam * kThreads * 16;
    const int vec4 = pair ? 4 : 8;
    const int cap_cols = kThreads * vec4 * 4;
    const int ctas_per_sm = pair ? 2 : 1;
    int capacity = sms * ctas_per_sm;
    if (capacity > 1024) capacity = 1024;
    RowPlan best{0, 0, 0, vec4, ctas_per_sm};
    double best_cost = 0.0;
    const int g_min = (vocab + cap_cols - 1) / cap_cols;
    for (int g = g_min; g <= kMaxTeam && g <= capacity; ++g) {
        int chunk = (vocab + g - 1) / g;
        chunk = (chunk + 3) & ~3;
        if ((vocab + chunk - 1) / chunk != g) continue;  // a member would be empty
        int64_t teams = capacity / g;
        if (teams > rows) teams = rows;
        if (teams < 1) continue;
        const double cost = static_cast<double>((rows + teams - 1) / teams) * chunk;
        if (best.team == 0 || cost < best_cost) {
            best = RowPlan{g, chunk, static_cast<int>(teams), vec4, ctas_per_sm};
            best_cost = cost;
        }
    }
    return best;
}

// ------------------------------------------------------ element helpers

__device__ __forceinline__ float comp(const float4& v, int q) {
    return q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w;
}

// 2^x on the special-function unit (non-flushing: subnormal results kept).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ------------------------------------------------ the temperature quotient

// x / t, rounded to nearest even, for one temperature t > 0 and many x.
// y = RN(1/t) once per row; per element q0 = x*y, then two corrections
// q <- q + (x - q*t)*y with the remainder taken exactly by an FMA
// (Markstein's scheme: the first correction makes q a faithful rounding of
// x/t, the second, with y the correctly rounded reciprocal, the correctly
// rounded quotient). A power-of-two t is a single exact multiplication and
// t == 1 is the identity. The FMA sequence turns an infinite x into NaN;
// `exact` maps +-inf to itself (x/t = x for finite t > 0), the row kernels
// treat NaN like -inf instead.
struct ScaledQuotient {
    enum Mode { kIdentity = 0, kScale = 1, kDivide = 2 };
    float t;
    float y;
    int mode;

    __device__ static ScaledQuotient of(float t) {
        ScaledQuotient q;
        q.t = t;
        q.y = __frcp_rn(t);
        const uint32_t b = __float_as_uint(t);
        const uint32_t e = (b >> 23) & 0xFFu;
        if (t == 1.0f) q.mode = kIdentity;
        else if ((b & 0x007FFFFFu) == 0 && e > 1 && e < 253) q.mode = kScale;
        else q.mode = kDivide;
        return q;
    }

    __device__ __forceinline__ float divide(float x) const {
        float q = x * y;
        float r = fmaf(-q, t, x);
        q = fmaf(r, y, q);
        r = fmaf(-q, t, x);
        return fmaf(r, y, q);
    }

    // Where the corrections are exact: the quotient and the dividend both
    // well inside the normal range, so that q*t, x*y and the remainder
    // x - q*t neither overflow nor underflow (a subnormal remainder loses
    // the bits the second correction needs).
    __device__ __forceinline__ static bool fast_ok(float x, float q) {
        const float ax = fabsf(x), aq = fabsf(q);
        return ax >= 0x1p-96f && ax <= 0x1p96f && aq >= 0x1p-100f && aq <= 0x1p100f;
    }

    // The quotient for every x: infinities map to themselves and quotients
    // outside the fast range take the IEEE division.
    __device__ __forceinline__ float exact(float x) const {
        if (mode == kIdentity) return x;
        if (mode == kScale) return x * y;
        if (fabsf(x) == INFINITY) return x;
        const float q = divide(x);
        return fast_ok(x, q) ? q : __fdiv_rn(x, t);
    }
};

}  // namespace drs
