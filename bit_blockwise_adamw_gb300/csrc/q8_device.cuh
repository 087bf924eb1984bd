// q8_device.cuh -- device-side building blocks of the step kernels: bf16 bit
// conversions, Philox4x32-10, stochastic rounding, the fp32 AdamW element
// update and the cell-table code search.
#pragma once

#include "q8_internal.h"

namespace q8 {

// ---------------------------------------------------------------- bf16 bits
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ---------------------------------------------------------------- Philox
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of
// (c0,c1,c2,c3) -> (hi(B*c2)^c1^k0, lo(B*c2), hi(A*c0)^c3^k1, lo(A*c0)) with
// the key advanced by the Weyl increments between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                               uint32_t k0, uint32_t k1)
{
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint32_t lo0 = 0xD2511F53u * c0;
        const uint32_t hi0 = __umulhi(0xD2511F53u, c0);
        const uint32_t lo1 = 0xCD9E8D57u * c2;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2);
        c0 = hi1 ^ c1 ^ k0;
        c1 = lo1;
        c2 = hi0 ^ c3 ^ k1;
        c3 = lo0;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return make_uint4(c0, c1, c2, c3);
}

// Draws of the eight elements E .. E+7 on Philox stream `sid`.  Element E
// takes half (E & 1) of word (E >> 1) & 3 of the call with counter
// (lo32(E/8), sid, step, hi32(E/8)).  Output word j holds the draws of
// elements E+2j (low half) and E+2j+1 (high half).  When E is not a multiple
// of 8 the eight draws span two calls; the shift `E & 7` is uniform across a
// tensor, so the branches below do not diverge inside a warp.
__device__ __forceinline__ void draws8(uint64_t E, uint32_t sid, const Scalars& s, uint32_t r[4])
{
    const uint64_t grp = E >> 3;
    const uint32_t sh = static_cast<uint32_t>(E) & 7u;
    const uint4 a = philox4x32_10(static_cast<uint32_t>(grp), sid, s.step,
                                  static_cast<uint32_t>(grp >> 32), s.k0, s.k1);
    if (sh == 0) {
        r[0] = a.x; r[1] = a.y; r[2] = a.z; r[3] = a.w;
        return;
    }
    const uint64_t g2 = grp + 1;
    const uint4 b = philox4x32_10(static_cast<uint32_t>(g2), sid, s.step,
                                  static_cast<uint32_t>(g2 >> 32), s.k0, s.k1);
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
// and keep the top half; NaN becomes 0x7FC0.  Returns the 32-bit pattern whose
// top half is the bf16 result (so two results pack with one byte permute).
__device__ __forceinline__ uint32_t sr_hi(float x, uint32_t r16)
{
    const uint32_t u = __float_as_uint(x) + r16;
    return (x != x) ? 0x7FC00000u : u;
}

__device__ __forceinline__ uint32_t rne_hi(float x)
{
    const uint32_t u = __float_as_uint(x);
    return (x != x) ? 0x7FC00000u : u + 0x7FFFu + ((u >> 16) & 1u);
}

// Top halves of a and b -> (b_hi << 16) | a_hi.
__device__ __forceinline__ uint32_t pack_hi(uint32_t a, uint32_t b) { return __byte_perm(a, b, 0x7632); }

// Round eight fp32 values to bf16 and pack them into four words.
__device__ __forceinline__ void round8(const float x[8], const uint32_t r[4], bool sr, uint32_t out[4])
{
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t lo = sr ? sr_hi(x[2 * j], r[j] & 0xFFFFu) : rne_hi(x[2 * j]);
        const uint32_t hi = sr ? sr_hi(x[2 * j + 1], r[j] >> 16) : rne_hi(x[2 * j + 1]);
        out[j] = pack_hi(lo, hi);
    }
}

// ---------------------------------------------------------------- AdamW
// One element, fp32, every operation rounded on its own (no contraction):
//   m = b1*m + (1-b1)*g;  v = b2*v + (1-b2)*g*g;
//   p = p*decay - a_t * (m / (sqrt(v) + eps_t))
__device__ __forceinline__ float adamw(const Scalars& s, float g, float p, float& m, float& v)
{
    const float mn = __fadd_rn(__fmul_rn(s.b1, m), __fmul_rn(s.omb1, g));
    const float vn = __fadd_rn(__fmul_rn(s.b2, v), __fmul_rn(s.omb2, __fmul_rn(g, g)));
    const float den = __fadd_rn(__fsqrt_rn(vn), s.eps_t);
    const float ratio = __fdiv_rn(mn, den);
    m = mn;
    v = vn;
    return __fsub_rn(__fmul_rn(p, s.decay), __fmul_rn(s.step_size, ratio));
}

// ---------------------------------------------------------------- search
// Code of a normalised value x: the number of codebook midpoints strictly
// below clamp(x, -1, 1), read from the cell table (see q8_internal.h).
template <int L, int kCellsPerSign>
__device__ __forceinline__ uint32_t cell_code(uint32_t u, const uint32_t* cells)
{
    const uint32_t a = min(u & 0x7FFFFFFFu, 0x3F800000u);        // |x| clamped to 1
    const int t = static_cast<int>(a) - ((127 - L) << 23);
    const int cell = max((t >> kCellShift) + 1, 0);
    const uint32_t neg = static_cast<uint32_t>(static_cast<int>(u) >> 31);
    const uint32_t e = cells[cell + (neg & static_cast<uint32_t>(kCellsPerSign))];
    const uint32_t xs = (a ^ neg) << 16;                          // low 16 bits, complemented if x < 0
    return (e & 0xFFu) + (xs > e ? 1u : 0u);
}

__device__ __forceinline__ uint32_t code_signed(float x, const uint32_t* cells)
{
    return cell_code<kSignedL, kCellsSigned>(__float_as_uint(x), cells);
}

// Unsigned book: negative x (and -0) code as +0; only the non-negative half
// of the table exists.
__device__ __forceinline__ uint32_t code_unsigned(float x, const uint32_t* cells)
{
    const uint32_t u = static_cast<uint32_t>(max(static_cast<int>(__float_as_uint(x)), 0));
    return cell_code<kUnsignedL, 0>(u, cells);
}

// ---------------------------------------------------------------- misc
__device__ __forceinline__ float warp_max(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xFFFFFFFFu, x, o));
    return x;
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
