// q8_device.cuh -- device-side building blocks of the step kernels: bf16 bit
// conversions, Philox4x32-10, stochastic rounding, the fp32 AdamW element
// update (on pairs, with Blackwell's packed fp32x2 instructions) and the
// cell-table code search.
#pragma once

#include "q8_internal.h"

namespace q8 {

// ---------------------------------------------------------------- bf16 bits
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
// The two bf16 values of one word as (low element, high element).
__device__ __forceinline__ float2 bf16x2(uint32_t w) { return make_float2(bf16lo(w), bf16hi(w)); }
// The same, the low half moved up by a multiply with two16 = 65536 passed in
// from the host (an integer multiply-add, on the FMA pipe) instead of a shift.
__device__ __forceinline__ float2 bf16x2_fma(uint32_t w, uint32_t two16)
{
    return make_float2(__uint_as_float(w * two16), bf16hi(w));
}

// ---------------------------------------------------------------- Philox
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of
// (c0,c1,c2,c3) -> (hi(B*c2)^c1^k0, lo(B*c2), hi(A*c0)^c3^k1, lo(A*c0)), the
// round keys taken from the host-formed schedule.
__device__ __forceinline__ uint4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                               const PhiloxKey& k)
{
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint32_t lo0 = 0xD2511F53u * c0;
        const uint32_t hi0 = __umulhi(0xD2511F53u, c0);
        const uint32_t lo1 = 0xCD9E8D57u * c2;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2);
        c0 = hi1 ^ c1 ^ k.kx[round];
        c1 = lo1;
        c2 = hi0 ^ c3 ^ k.ky[round];
        c3 = lo0;
    }
    return make_uint4(c0, c1, c2, c3);
}

// Draws of the eight elements E .. E+7 on Philox stream `sid`.  Element E
// takes half (E & 1) of word (E >> 1) & 3 of the call with counter
// (lo32(E/8), sid, step, hi32(E/8)).  Output word j holds the draws of
// elements E+2j (low half) and E+2j+1 (high half).  When E is not a multiple
// of 8 the eight draws span two calls; the shift `E & 7` is uniform across a
// tensor, so the branches below do not diverge inside a warp.
__device__ __forceinline__ void draws8(uint64_t E, uint32_t sid, const PhiloxKey& k, uint32_t r[4])
{
    const uint64_t grp = E >> 3;
    const uint32_t sh = static_cast<uint32_t>(E) & 7u;
    const uint4 a = philox4x32_10(static_cast<uint32_t>(grp), sid, k.step, static_cast<uint32_t>(grp >> 32), k);
    if (sh == 0) {
        r[0] = a.x; r[1] = a.y; r[2] = a.z; r[3] = a.w;
        return;
    }
    const uint64_t g2 = grp + 1;
    const uint4 b = philox4x32_10(static_cast<uint32_t>(g2), sid, k.step, static_cast<uint32_t>(g2 >> 32), k);
    uint32_t w0 = a.x, w1 = a.y, w2 = a.z, w3 = a.w, w4 = b.x, w5 = b.y, w6 = b.z, w7 = b.w;
    if (sh & 4u) { w0 = w2; w1 = w3; w2 = w4; w3 = w5; w4 = w6; w5 = w7; }
    if (sh & 2u) { w0 = w1; w1 = w2; w2 = w3; w3 = w4; w4 = w5; }
    if (sh & 1u) {
        w0 = __funnelshift_r(w0, w1, 16);
        w1 = __funnelshift_r(w1, w2, 16);
        w2 = __funnelshift_r(w2, w3, 16);
        w3 = __funnelshift_r(w3, w4, 16);
    }
    r[0] = w0; r[1] = w1; r[2] = w2; r[3] = w3;
}

// ---------------------------------------------------------------- rounding
// Stochastic rounding fp32 -> bf16 ("Stochastic rounding support for 8-bit
// optimizers", feature request): add a uniform 16-bit draw to the bit pattern
// and keep the top half; NaN becomes 0x7FC0.  These return the 32-bit pattern
// whose top half is the bf16 result, so two results pack with one permute.
//
// NaN: the fp32 values rounded here are results of GPU arithmetic, whose NaN
// is the canonical 0x7FFFFFFF (the largest positive pattern), so a signed
// integer min with 0x7FC00000 maps it to the quiet NaN 0x7FC00000 (whose
// top half survives the add) and leaves every number and infinity alone.
__device__ __forceinline__ uint32_t quiet_nan(uint32_t u)
{
    return static_cast<uint32_t>(min(static_cast<int>(u), 0x7FC00000));
}

__device__ __forceinline__ uint32_t sr_hi(float x, uint32_t r16)
{
    return quiet_nan(__float_as_uint(x)) + r16;
}

__device__ __forceinline__ uint32_t rne_hi(float x)
{
    const uint32_t u = quiet_nan(__float_as_uint(x));
    return u + 0x7FFFu + ((u >> 16) & 1u);
}

// Top halves of a and b -> (b_hi << 16) | a_hi.
__device__ __forceinline__ uint32_t pack_hi(uint32_t a, uint32_t b) { return __byte_perm(a, b, 0x7632); }

// The same for a pair known to hold no NaN (infinities are fine: the add
// cannot carry out of them), without the quieting.
template <bool SR>
__device__ __forceinline__ uint32_t round2_num(float2 x, uint32_t r)
{
    const uint32_t ux = __float_as_uint(x.x), uy = __float_as_uint(x.y);
    if constexpr (SR) return pack_hi(ux + (r & 0xFFFFu), uy + (r >> 16));
    else return pack_hi(ux + 0x7FFFu + ((ux >> 16) & 1u), uy + 0x7FFFu + ((uy >> 16) & 1u));
}

// Round a pair to bf16 and pack it into one word (draws in r: low half for
// the first element, high half for the second).
template <bool SR>
__device__ __forceinline__ uint32_t round2(float2 x, uint32_t r)
{
    if constexpr (SR) return pack_hi(sr_hi(x.x, r & 0xFFFFu), sr_hi(x.y, r >> 16));
    else return pack_hi(rne_hi(x.x), rne_hi(x.y));
}

// ---------------------------------------------------------------- AdamW
// The fp32 update, with each multiply-add fused (one rounding) and every
// other operation rounded on its own:
//   m = fma(b1, m, (1-b1)*g);  v = fma(b2, v, (1-b2)*(g*g));
//   p = fma(-a_t, m / (sqrt(v) + eps_t), p*decay)
// Pairs use the packed fp32x2 instructions (per lane identical to the scalar
// _rn operations).  Every product feeds an explicit fma or nothing, so the
// compiler has no multiply-add left to contract; the square root stays
// scalar, the division is packed where it is provably exact (below).
__device__ __forceinline__ float2 splat(float x) { return make_float2(x, x); }

// The moment updates of a pair: m = fma(b1, m, (1-b1)*g), v = fma(b2, v, (1-b2)*g*g).
__device__ __forceinline__ void moments2(const Scalars& s, float2 g, float2& m, float2& v)
{
    m = __ffma2_rn(splat(s.b1), m, __fmul2_rn(splat(s.omb1), g));
    v = __ffma2_rn(splat(s.b2), v, __fmul2_rn(splat(s.omb2), __fmul2_rn(g, g)));
}

// ---------------------------------------------------------------- division
// Correctly rounded quotients on the packed fp32x2 unit.  y = RN(1/d) comes
// from the hardware's approximate reciprocal and one Newton-Raphson step,
// y = y0 + y0*(1 - d*y0) with each multiply-add fused; this equals the IEEE
// reciprocal for every normal d whose reciprocal is normal (checked over all
// of them, q8_selftest_sqrt_div).  Then Markstein's correction ("Computation
// of elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990): q0 = RN(m*y), r = RN(m - d*q0) (one fma),
// q = RN(q0 + r*y) (one fma) is RN(m/d) when y = RN(1/d) and no intermediate
// leaves the normal range.  Callers use it only inside the kDiv* bounds and
// fall back to the IEEE division otherwise.
constexpr float kDivMinM = 0x1p-90f;      // |m| at least this (and nonzero: the sign of 0)
constexpr float kDivMaxM = 0x1p26f;       // |m| at most this
constexpr float kDivMaxV = 0x1p40f;       // v at most this, so sqrt(v) <= 2^20
// with eps_t in [2^-100, 2^20] (host flag Scalars::fast_div): d in [2^-100, 2^21],
// 1/d normal, |q| in [2^-111, 2^126], the remainder's scale |m|*2^-23 normal.

__device__ __forceinline__ float rcp_approx(float d)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(d));
    return y;
}

__device__ __forceinline__ float2 neg2(float2 x) { return make_float2(-x.x, -x.y); }

// RN(1/d) of a pair (d normal with a normal reciprocal).
__device__ __forceinline__ float2 recip2(float2 d)
{
    const float2 y0 = make_float2(rcp_approx(d.x), rcp_approx(d.y));
    const float2 e = __ffma2_rn(neg2(d), y0, make_float2(1.0f, 1.0f));
    return __ffma2_rn(y0, e, y0);
}

// RN(1/x) of one value: the Newton-corrected approximation where it is exact
// (x normal with a normal reciprocal), the IEEE reciprocal elsewhere (0, tiny,
// huge and non-finite x).  Used once per block, so the branch is uniform.
__device__ __forceinline__ float recip_rn(float x)
{
    if (x >= 0x1p-126f && x < 0x1p126f) {
        const float y0 = rcp_approx(x);
        return __fmaf_rn(y0, __fmaf_rn(-x, y0, 1.0f), y0);
    }
    return __frcp_rn(x);
}

// RN(m/d) of a pair inside the bounds above.
__device__ __forceinline__ float2 div2_rn(float2 m, float2 d)
{
    const float2 y = recip2(d);
    const float2 q0 = __fmul2_rn(m, y);
    const float2 r = __ffma2_rn(neg2(d), q0, m);
    return __ffma2_rn(r, y, q0);
}

// m / (sqrt(v) + eps_t) of a pair, given sqrt(v).
__device__ __forceinline__ float2 ratio2(const Scalars& s, float2 m, float2 root)
{
    const float2 den = __fadd2_rn(root, splat(s.eps_t));
    return make_float2(__fdiv_rn(m.x, den.x), __fdiv_rn(m.y, den.y));
}

// p*decay - a_t*ratio of a pair.
__device__ __forceinline__ float2 step2(const Scalars& s, float2 p, float2 ratio)
{
    return __ffma2_rn(splat(-s.step_size), ratio, __fmul2_rn(p, splat(s.decay)));
}

// RN(sqrt(v)) of a pair: the hardware's approximate reciprocal square root
// y and one Newton-Raphson (Heron) correction, s = s0 + (v - s0*s0)*(y/2)
// with s0 = RN(v*y), each multiply-add fused.  Equal to the IEEE square root
// for every normal v >= 2^-102 (checked over all of them,
// q8_selftest_sqrt_div); the callers use it for v in [kSqrtMinV, kDivMaxV].
constexpr float kSqrtMinV = 0x1p-100f;

__device__ __forceinline__ float rsqrt_approx(float v)
{
    float y;
    asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(v));
    return y;
}

__device__ __forceinline__ float2 sqrt2_rn(float2 v)
{
    const float2 y = make_float2(rsqrt_approx(v.x), rsqrt_approx(v.y));
    const float2 s0 = __fmul2_rn(v, y);
    const float2 h = __fmul2_rn(make_float2(0.5f, 0.5f), y);
    const float2 r = __ffma2_rn(neg2(s0), s0, v);
    return __ffma2_rn(r, h, s0);
}

// The same ratio with the packed division (only inside the bounds above).
__device__ __forceinline__ float2 ratio2_fast(const Scalars& s, float2 m, float2 root)
{
    return div2_rn(m, __fadd2_rn(root, splat(s.eps_t)));
}

// The fast mode's m / (sqrt(v) + eps_t) of a pair: the hardware's approximate
// square root and reciprocal (flush-to-zero forms, one instruction each, each
// within 2^-21 relative error over every normal input, measured by
// q8_selftest_sqrt_div), then one packed add and one packed multiply.  With
// the roundings of the add and the multiply, the quotient q is within 2^-19
// relative error of the correctly rounded one.  Callers use it when
// Scalars::approx is set: eps_t in [2^-36, 2^20] keeps the denominator normal
// and makes the square root of a subnormal v (flushed to 0) fall below half
// an ulp of eps_t, as the exact step rounds it; infinite or NaN v gives 0 or
// NaN as the division does.
//
// It feeds only the parameter update P = fma(-a_t, q, p*decay), never m or
// v, so codes, absmax and BF16 moments are those of the exact step.  P itself
// can move by a_t * 2^-19 * |q| plus its own rounding: when the update nearly
// cancels p*decay that is many BF16 ulps of the small P.  So the callers redo
// on the exact path every element unless |P| >= |q| * a_t * 2^-9
// (Scalars::cancel; the AdamW kernel checks each element, the BF16-state
// kernel the thread's smallest |P| against its largest |q|).  Past that bound
// the two P lie fewer than 2^15 fp32 values apart, with the same sign, so
// after the same 16-bit stochastic-rounding draw (or rounding to nearest
// even) their BF16 results differ by one ulp at most.
__device__ __forceinline__ float sqrt_approx(float v)
{
    float y;
    asm("sqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(v));
    return y;
}

__device__ __forceinline__ float2 ratio2_approx(const Scalars& s, float2 m, float2 v)
{
    const float2 den = __fadd2_rn(make_float2(sqrt_approx(v.x), sqrt_approx(v.y)), splat(s.eps_t));
    return __fmul2_rn(m, make_float2(rcp_approx(den.x), rcp_approx(den.y)));
}

// The parameter update of a pair given sqrt(v): p*decay - a_t*(m/(sqrt(v)+eps_t)).
__device__ __forceinline__ float2 param2(const Scalars& s, float2 p, float2 m, float2 root)
{
    return step2(s, p, ratio2(s, m, root));
}

// Scalar form (same rounding), for the small-tensor kernel.
__device__ __forceinline__ float adamw(const Scalars& s, float g, float p, float& m, float& v)
{
    const float mn = __fmaf_rn(s.b1, m, __fmul_rn(s.omb1, g));
    const float vn = __fmaf_rn(s.b2, v, __fmul_rn(s.omb2, __fmul_rn(g, g)));
    const float ratio = __fdiv_rn(mn, __fadd_rn(__fsqrt_rn(vn), s.eps_t));
    m = mn;
    v = vn;
    return __fmaf_rn(-s.step_size, ratio, __fmul_rn(p, s.decay));
}

// ---------------------------------------------------------------- search
// Code of a normalised value: the number of codebook midpoints strictly
// below clamp(y, -1, 1), y = m * RN(1/absmax), read from the cell table
// (layout in q8_internal.h).  The callers form |y| clamped to [0, 1] with one
// saturating multiply (mul.sat: NaN gives 0), so the magnitude needs no
// further clamp, and take the sign from m.  The result is correct in its low
// byte; codes are packed with byte permutes, which ignore the upper bits.
__device__ __forceinline__ uint32_t sat_mul_bits(float x, float s)
{
    float r;
    asm("mul.rn.sat.f32 %0, %1, %2;" : "=f"(r) : "f"(x), "f"(s));
    return __float_as_uint(r);
}

// Four codes (low bytes of q0..q3) -> one word, q0 in the lowest byte.
__device__ __forceinline__ uint32_t pack4(uint32_t q0, uint32_t q1, uint32_t q2, uint32_t q3)
{
    return __byte_perm(__byte_perm(q0, q1, 0x0040), __byte_perm(q2, q3, 0x0040), 0x5410);
}

// m scaled by inv (= RN(1/absmax) > 0): code in the signed book.  a holds the
// bits of min(|m|*inv, 1) (one saturating multiply).  The table counts, per
// magnitude cell, the positive midpoints (indices 127..253) below the cell and
// holds the low bits of the one inside it.  By the odd symmetry of the signed
// book, m > 0 takes code 127 + #{positive midpoints < |y|} and m < 0 takes
// 127 - #{positive midpoints <= |y|}.  count_signed_scaled returns that count
// (in its low byte): the comparison key carries 0xFF00 in its low half for
// m < 0 (above any base count, below the marker of a cell without a
// midpoint), which turns "<" into "<=".  signed_codes4 applies the signs to
// four counts at once.
__device__ __forceinline__ uint32_t count_signed_scaled(float m, float inv, const uint32_t* cells)
{
    const uint32_t a = sat_mul_bits(fabsf(m), inv);
    const int cell = __viaddmax_s32(static_cast<int>(a >> kCellShift), kSignedCellBias, 0);
    const uint32_t e = cells[cell];
    // key bytes, high to low: a.b1, a.b0, the sign of m replicated, the sign of
    // a replicated (0, as a >= 0): (a << 16) | (m < 0 ? 0xFF00 : 0)
    uint32_t key;
    asm("prmt.b32 %0, %1, %2, 0x10FB;" : "=r"(key) : "r"(a), "r"(__float_as_uint(m)));
    return e + (key > e ? 1u : 0u);
}

// Signed codes of four values from their counts c0..c3 (low bytes) and their
// signs: byte i is 127 + c_i for m_i >= 0 and 127 - c_i for m_i < 0.  With C
// the packed counts and S the packed sign bytes (0xFF for m_i < 0), byte i of
// (C ^ S) - S is +c_i or -c_i, and as every byte of the result lies in
// [0, 254], the one 32-bit sum 0x7F7F7F7F + (C ^ S) - S has exactly those
// bytes (no carry or borrow crosses a byte).
__device__ __forceinline__ uint32_t signed_codes4(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, float m0,
                                                  float m1, float m2, float m3)
{
    const uint32_t C = pack4(c0, c1, c2, c3);
    uint32_t s01, s23, S;
    // byte 0 <- sign of byte 3 (m0's top byte) replicated, byte 1 <- sign of byte 7 (m1's)
    asm("prmt.b32 %0, %1, %2, 0x00FB;" : "=r"(s01) : "r"(__float_as_uint(m0)), "r"(__float_as_uint(m1)));
    asm("prmt.b32 %0, %1, %2, 0x00FB;" : "=r"(s23) : "r"(__float_as_uint(m2)), "r"(__float_as_uint(m3)));
    S = __byte_perm(s01, s23, 0x5410);
    return 0x7F7F7F7Fu + (C ^ S) - S;
}

// The signed code of one value (low byte of the result).
__device__ __forceinline__ uint32_t code_signed_scaled(float m, float inv, const uint32_t* cells)
{
    const uint32_t c = count_signed_scaled(m, inv, cells);
    const uint32_t s = static_cast<uint32_t>(static_cast<int>(__float_as_uint(m)) >> 31) | 1u;
    return c * s + 127u;
}

// a: bits of a value in [0, 1] (unsigned book).
__device__ __forceinline__ uint32_t code_unsigned_mag(uint32_t a, const uint32_t* cells)
{
    const int cell = __viaddmax_s32(static_cast<int>(a >> kCellShift), kUnsignedCellBias, 0);
    const uint32_t e = cells[cell];
    return e + ((a << 16) > e ? 1u : 0u);
}

// v scaled by inv: code in the unsigned book (negative values code as 0).
__device__ __forceinline__ uint32_t code_unsigned_scaled(float v, float inv, const uint32_t* cells)
{
    return code_unsigned_mag(sat_mul_bits(v, inv), cells);
}

// Byte j (0..3) of w, zero-extended.
__device__ __forceinline__ uint32_t byte_of(uint32_t w, int j) { return __byte_perm(w, 0u, 0x4440 | j); }

// ---------------------------------------------------------------- misc
__device__ __forceinline__ float min3(float a, float b, float c)
{
    float r;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ float max3(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}


// Ask the L2 to fetch [p, p + bytes) from DRAM now: a hint that completes
// asynchronously and is never waited for.  bytes must be a multiple of 16.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Streaming loads/stores: every byte of the step is touched once.
__device__ __forceinline__ uint4 ld_stream16(const void* p)
{
    return __ldcs(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ uint2 ld_stream8(const void* p)
{
    return __ldcs(reinterpret_cast<const uint2*>(p));
}
__device__ __forceinline__ void st_stream16(void* p, uint4 v) { __stcs(reinterpret_cast<uint4*>(p), v); }
__device__ __forceinline__ void st_stream8(void* p, uint2 v) { __stcs(reinterpret_cast<uint2*>(p), v); }

}  // namespace q8
