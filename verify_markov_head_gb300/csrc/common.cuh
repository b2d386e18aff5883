// common.cuh -- device helpers shared by the DSpark kernels: the counter-based
// generator, the Gumbel transform, the mergeable sampling / log-sum-exp state,
// and the workspace layout.
//
// Random numbers follow the stream definition stated in include/dspark.h:
// Philox4x32-10 as specified by Salmon, Moraes, Dror and Shaw ("Parallel
// Random Numbers: As Easy as 1, 2, 3", SC'11, section 3), written here from
// that specification.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dspark.h"
#include "internal.h"

namespace dspark {

// ---------------------------------------------------------------- Philox4x32-10
struct Philox {
    static constexpr uint32_t kM0 = 0xD2511F53u, kM1 = 0xCD9E8D57u;   // round multipliers
    static constexpr uint32_t kW0 = 0x9E3779B9u, kW1 = 0xBB67AE85u;   // key increments
};

// 32 x 32 -> 64-bit product; one wide multiply yields both halves.
__device__ __forceinline__ uint64_t mul_wide(uint32_t a, uint32_t b) {
    uint64_t r;
    asm("mul.wide.u32 %0, %1, %2;" : "=l"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint4 philox_round(uint4 c, uint32_t k0, uint32_t k1) {
    const uint64_t p0 = mul_wide(Philox::kM0, c.x);
    const uint64_t p1 = mul_wide(Philox::kM1, c.z);
    return make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ k0, (uint32_t)p1, (uint32_t)(p0 >> 32) ^ c.w ^ k1, (uint32_t)p0);
}

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int i = 0; i < 10; ++i) {
        if (i) { k0 += Philox::kW0; k1 += Philox::kW1; }
        c = philox_round(c, k0, k1);
    }
    return c;
}

// The four words for columns 4*quad .. 4*quad+3 of one (row, domain) stream.
struct Stream {
    uint32_t k0, k1, row, step_lo, dom_hi;
    __device__ __forceinline__ Stream(uint64_t seed, uint64_t step, uint32_t domain, uint32_t row_)
        : k0((uint32_t)seed), k1((uint32_t)(seed >> 32)), row(row_), step_lo((uint32_t)step),
          dom_hi(domain + 4u * (uint32_t)(step >> 32)) {}
    __device__ __forceinline__ uint4 quad(uint32_t q) const {
        return philox4x32_10(make_uint4(q, row, step_lo, dom_hi), k0, k1);
    }
    __device__ __forceinline__ uint32_t word(uint32_t col) const {
        const uint4 w = quad(col >> 2);
        const uint32_t s = col & 3u;
        return s == 0 ? w.x : s == 1 ? w.y : s == 2 ? w.z : w.w;
    }
};

// The same stream with the ten round keys computed once, for loops that draw
// many quads of one row.
// Only the first counter word varies along a row, so half of the first
// round (the product of the third word and its XOR with the second word and
// key) is the same for every quad and is formed once here.
struct StreamRK {
    uint32_t rk0[10], rk1[10];
    uint32_t r1x, r1y, dom_k1;    // round 1: hi(M1*step_lo) ^ row ^ k0, lo(M1*step_lo), dom_hi ^ k1
    __device__ __forceinline__ StreamRK(uint64_t seed, uint64_t step, uint32_t domain, uint32_t row) {
        uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
#pragma unroll
        for (int i = 0; i < 10; ++i) {
            rk0[i] = k0; rk1[i] = k1;
            k0 += Philox::kW0; k1 += Philox::kW1;
        }
        const uint64_t p1 = mul_wide(Philox::kM1, (uint32_t)step);
        r1x = (uint32_t)(p1 >> 32) ^ row ^ rk0[0];
        r1y = (uint32_t)p1;
        dom_k1 = (domain + 4u * (uint32_t)(step >> 32)) ^ rk1[0];
    }
    __device__ __forceinline__ uint4 quad(uint32_t q) const {
        const uint64_t p0 = mul_wide(Philox::kM0, q);
        uint4 c = make_uint4(r1x, r1y, (uint32_t)(p0 >> 32) ^ dom_k1, (uint32_t)p0);
#pragma unroll
        for (int i = 1; i < 10; ++i) c = philox_round(c, rk0[i], rk1[i]);
        return c;
    }
};

// u = (2*(x >> 9) + 1) * 2^-24, exact in binary32, strictly inside (0, 1):
// with j = x >> 9, the float 1 + j*2^-23 (exponent 127, mantissa j) minus
// 1 - 2^-24 is exactly (2j + 1) * 2^-24.
constexpr float kOneMinusHalfUlp = 0.99999994039535522f;   // 1 - 2^-24
__device__ __forceinline__ float uniform_of(uint32_t x) {
    return __uint_as_float((x >> 9) | 0x3f800000u) - kOneMinusHalfUlp;
}
// 1 - u, exactly: the same construction on the complemented top 23 bits.
__device__ __forceinline__ float one_minus_uniform_of(uint32_t x) {
    return __uint_as_float((~x >> 9) | 0x3f800000u) - kOneMinusHalfUlp;
}

// log2(x) on the special-function unit, flush-to-zero form (the arguments
// here are normal numbers >= 2^-24, so no subnormal fix-up is needed).
__device__ __forceinline__ float fast_log2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Standard Gumbel variate G = -ln(E), E = -ln(u).
//   E: for u <= 7/8, -ln2 * log2(u) with the hardware log2 (absolute error
//      <= 2^-22 on [1/2, 2], 2 ulp elsewhere, so E keeps ~1e-6 relative
//      accuracy where |log2 u| >= 0.19); for w = 1 - u < 1/8, the Taylor
//      series -ln(1 - w) = sum_{n>=1} w^n / n to n = 8 (next term below
//      7e-9 relative).  w is exact, so E stays accurate as u -> 1, where
//      the largest variates (the likely winners) come from.
//   G: -ln2 * log2(E), absolute error <= 2e-7.
// Overall |G - exact| stays near 1e-6; the oracle computes G in binary64.
constexpr float kLn2 = 0.69314718055994531f;
__device__ __forceinline__ float gumbel_of(uint32_t x) {
    const float u = uniform_of(x);
    const float w = one_minus_uniform_of(x);
    const float e_log = -kLn2 * fast_log2(u);
    float poly = fmaf(w, 0.125f, 0.142857143f);
    poly = fmaf(w, poly, 0.166666667f);
    poly = fmaf(w, poly, 0.2f);
    poly = fmaf(w, poly, 0.25f);
    poly = fmaf(w, poly, 0.333333333f);
    poly = fmaf(w, poly, 0.5f);
    poly = fmaf(w, poly, 1.0f);
    const float E = (w < 0.125f) ? w * poly : e_log;
    return -kLn2 * fast_log2(E);
}

// E2 = -log2(u) (the exponential variate -ln u in base-2 units), for the
// exponential-race form of Gumbel-max:
//   argmax_v z_v + G_v  =  argmin_v E_v * e^(-z_v)  =  argmin_v E2_v * 2^(-z_v*log2e),
// the same draw without the outer logarithm.  E2 takes the series
// -ln(1 - w) * log2e = sum_{n>=1} (log2e/n) w^n to n = 8 for w = 1 - u < 1/8
// (exact w, so E2 keeps its relative accuracy as u -> 1) and the hardware
// log2 elsewhere, as in gumbel_of.
__device__ __forceinline__ float exp2_variate_of(uint32_t x) {
    const float u = uniform_of(x);
    const float w = one_minus_uniform_of(x);
    const float e_log = -fast_log2(u);
    float poly = fmaf(w, 0.18033688011112042f, 0.20609929155556619f);   // log2e/8, log2e/7
    poly = fmaf(w, poly, 0.24044917348149389f);                          // log2e/6
    poly = fmaf(w, poly, 0.28853900817779268f);                          // log2e/5
    poly = fmaf(w, poly, 0.36067376022224085f);                          // log2e/4
    poly = fmaf(w, poly, 0.48089834696298783f);                          // log2e/3
    poly = fmaf(w, poly, 0.72134752044448170f);                          // log2e/2
    poly = fmaf(w, poly, 1.4426950408889634f);                           // log2e
    return (w < 0.125f) ? w * poly : e_log;
}

// 2^x on the special-function unit (relative error about 2^-22, subnormal
// results flushed to zero).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---------------------------------------------------------------- merge states
// Gumbel-max draw fused with a log-sum-exp: over a set of entries,
//   best = max (z_v + G_v), idx = its v (lowest v on ties), zb = z_idx
//          (best = -inf, idx = 2^31 - 1: no draw taken in the set),
//   lse  = log sum_v exp(z_v)  (-inf for an empty set).
// The two parts merge independently, so the log-sum-exp of a set does not
// depend on which entries a partial draw examined: a draw may skip entries
// that cannot win (screened against a bound found elsewhere) while the sum
// covers every entry.
struct DrawLse {
    float best;
    int idx;
    float zb;
    float lse;
};

static_assert(sizeof(DrawLse) == kDrawLseBytes, "the workspace layout counts 16 bytes per partial state");

__device__ __forceinline__ DrawLse drawlse_empty() { return DrawLse{-INFINITY, 0x7fffffff, 0.f, -INFINITY}; }

__device__ __forceinline__ bool wins(float sa, int ia, float sb, int ib) {
    return sa > sb || (sa == sb && ia < ib);
}

// log(e^x + e^y), with -inf as the empty sum.  log(1 + w) for w in (0, 1]
// through the hardware log2 of 1 + w: absolute error about 1e-7 (the rounding
// of 1 + w loses at most w * 2^-24 of it).
__device__ __forceinline__ float log_add_exp(float x, float y) {
    const float m = fmaxf(x, y), n = fminf(x, y);
    if (n == -INFINITY) return m;
    float l2;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(l2) : "f"(1.f + __expf(n - m)));
    return fmaf(l2, 0.69314718055994531f, m);
}

__device__ __forceinline__ DrawLse drawlse_merge(const DrawLse& a, const DrawLse& b) {
    DrawLse o = wins(b.best, b.idx, a.best, a.idx) ? b : a;
    o.lse = log_add_exp(a.lse, b.lse);
    return o;
}

__device__ __forceinline__ DrawLse shfl_xor(const DrawLse& a, int m) {
    DrawLse o;
    o.best = __shfl_xor_sync(0xffffffffu, a.best, m);
    o.idx = __shfl_xor_sync(0xffffffffu, a.idx, m);
    o.zb = __shfl_xor_sync(0xffffffffu, a.zb, m);
    o.lse = __shfl_xor_sync(0xffffffffu, a.lse, m);
    return o;
}

// Online log-sum-exp (running max reference) plus an optional Gumbel-max draw.
struct LseDraw {
    float m;     // running max of x
    float s;     // sum exp(x - m)
    float best;  // max (x + G) or -inf when no draw is taken
    int idx;
};

__device__ __forceinline__ LseDraw lsedraw_empty() { return LseDraw{-INFINITY, 0.f, -INFINITY, 0x7fffffff}; }

__device__ __forceinline__ LseDraw lsedraw_merge(const LseDraw& a, const LseDraw& b) {
    LseDraw o;
    if (b.m == -INFINITY) { o.m = a.m; o.s = a.s; }
    else if (a.m == -INFINITY) { o.m = b.m; o.s = b.s; }
    else if (a.m >= b.m) { o.m = a.m; o.s = a.s + b.s * __expf(b.m - a.m); }
    else { o.m = b.m; o.s = b.s + a.s * __expf(a.m - b.m); }
    if (wins(b.best, b.idx, a.best, a.idx)) { o.best = b.best; o.idx = b.idx; }
    else { o.best = a.best; o.idx = a.idx; }
    return o;
}

__device__ __forceinline__ LseDraw shfl_xor(const LseDraw& a, int m) {
    LseDraw o;
    o.m = __shfl_xor_sync(0xffffffffu, a.m, m);
    o.s = __shfl_xor_sync(0xffffffffu, a.s, m);
    o.best = __shfl_xor_sync(0xffffffffu, a.best, m);
    o.idx = __shfl_xor_sync(0xffffffffu, a.idx, m);
    return o;
}

// Two Gumbel-max draws over the same set (residual law and its fallback p).
struct Draw2 {
    float best_r; int idx_r;   // argmax log(max(0, p - q)) + G   (only where p > q)
    float best_p; int idx_p;   // argmax x_p + G                  (fallback law p)
};

__device__ __forceinline__ Draw2 draw2_empty() { return Draw2{-INFINITY, 0x7fffffff, -INFINITY, 0x7fffffff}; }

__device__ __forceinline__ Draw2 draw2_merge(const Draw2& a, const Draw2& b) {
    Draw2 o;
    if (wins(b.best_r, b.idx_r, a.best_r, a.idx_r)) { o.best_r = b.best_r; o.idx_r = b.idx_r; }
    else { o.best_r = a.best_r; o.idx_r = a.idx_r; }
    if (wins(b.best_p, b.idx_p, a.best_p, a.idx_p)) { o.best_p = b.best_p; o.idx_p = b.idx_p; }
    else { o.best_p = a.best_p; o.idx_p = a.idx_p; }
    return o;
}

__device__ __forceinline__ Draw2 shfl_xor(const Draw2& a, int m) {
    Draw2 o;
    o.best_r = __shfl_xor_sync(0xffffffffu, a.best_r, m);
    o.idx_r = __shfl_xor_sync(0xffffffffu, a.idx_r, m);
    o.best_p = __shfl_xor_sync(0xffffffffu, a.best_p, m);
    o.idx_p = __shfl_xor_sync(0xffffffffu, a.idx_p, m);
    return o;
}

// ---------------------------------------------------------------- loads
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(uint16_t x) { return __uint_as_float(((uint32_t)x) << 16); }

template <typename T> struct Vec4;
template <> struct Vec4<float> {
    __device__ __forceinline__ static float4 load(const float* p) { return *reinterpret_cast<const float4*>(p); }
    __device__ __forceinline__ static float4 load_stream(const float* p) {
        return __ldcs(reinterpret_cast<const float4*>(p));
    }
};
template <> struct Vec4<uint16_t> {
    __device__ __forceinline__ static float4 cvt(uint2 v) {
        return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u),
                           __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
    }
    __device__ __forceinline__ static float4 load(const uint16_t* p) {
        return cvt(*reinterpret_cast<const uint2*>(p));
    }
    __device__ __forceinline__ static float4 load_stream(const uint16_t* p) {
        return cvt(__ldcs(reinterpret_cast<const uint2*>(p)));
    }
};

// ---------------------------------------------------------------- status word
enum StatusBits : uint32_t {
    kBadToken = 1u << 0,     // a token id outside [0, V)
    kBadLength = 1u << 1,    // a verify length outside [0, gamma]
    kTimeout = 1u << 2,      // a bounded wait expired
    kBadInput = 1u << 3,     // a non-finite score or a temperature that is not positive and finite
};

__device__ __forceinline__ void raise_status(uint32_t* status, uint32_t bit) {
    if (status) atomicOr(status, bit);
}

// The bound on device waits that can block on another role or CTA: the
// workspace's value (dspark_workspace_set_wait_limit), 0 meaning the default
// of about 2 s at 2 GHz.  Drains of copies already issued keep their own
// fixed bounds: those copies always land.
constexpr long long kDefaultWaitCycles = 4000000000LL;
__device__ __forceinline__ long long wait_limit_of(const unsigned long long* w) {
    const unsigned long long v = w ? *w : 0ull;
    return v ? (long long)v : kDefaultWaitCycles;
}

// A bounded wait expired: the timeout bit, plus bit (8 + site) naming the
// wait that gave up (sites 0..23, see the kernel that raises it).
__device__ __forceinline__ void raise_timeout(uint32_t* status, int site) {
    if (status) atomicOr(status, kTimeout | (1u << (8 + (site & 15))));
}

}  // namespace dspark
