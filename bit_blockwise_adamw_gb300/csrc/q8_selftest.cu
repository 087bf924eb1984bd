// q8_selftest.cu -- device self-test of the packed square root and division
// used by the AdamW steps (q8_device.cuh, "division"), against CUDA's IEEE
// reciprocal, division and square root: every positive normal d with a normal
// reciprocal for y = RN(1/d), seeded pseudo-random quotients inside the bounds
// the steps check, and every normal v >= 2^-100 for the square root.  It also
// measures the largest relative error of the approximate square root and
// reciprocal of the fast mode (ratio2_approx), against double precision, over
// every normal input.
#include "q8_device.cuh"

namespace q8 {

namespace {

constexpr uint32_t kFirstD = 0x00800000u;      // 2^-126
constexpr uint32_t kEndD = 0x7E800000u;        // 2^126: 1/d is normal below this
constexpr int kPairsPerD = 2;
constexpr uint32_t kFirstV = 0x0D800000u;      // 2^-100
constexpr uint32_t kEndV = 0x7F800000u;        // +inf
constexpr uint32_t kFirstNormal = 0x00800000u; // 2^-126

// A 32-bit integer mix (xor-shift-multiply) for the pseudo-random pairs.
__device__ __forceinline__ uint32_t mix(uint32_t x)
{
    x ^= x >> 16;
    x *= 0x7FEB352Du;
    x ^= x >> 15;
    x *= 0x846CA68Bu;
    x ^= x >> 16;
    return x;
}

// A float with random mantissa and sign and a biased exponent in [lo, lo + span).
__device__ __forceinline__ float random_float(uint32_t h, uint32_t lo, uint32_t span, bool sign)
{
    const uint32_t e = lo + mix(h) % span;
    return __uint_as_float((h & (sign ? 0x807FFFFFu : 0x007FFFFFu)) | (e << 23));
}

__global__ void __launch_bounds__(256) selftest_kernel(unsigned long long* counts)
{
    unsigned long long bad_y = 0, bad_q = 0, pairs = 0;
    const uint32_t n = kEndD - kFirstD;
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const float d = __uint_as_float(kFirstD + i);
        const float2 y = recip2(make_float2(d, d));
        bad_y += __float_as_uint(y.x) != __float_as_uint(__frcp_rn(d));
        // pairs inside the bounds: m with |m| in [2^-90, 2^26], d' in [2^-100, 2^21]
#pragma unroll
        for (int j = 0; j < kPairsPerD; ++j) {
            const uint32_t h = mix(i * 2u + j + 0x9E3779B9u);
            const float m = random_float(h, 127 - 90, 90 + 26 + 1, true);
            const float dd = random_float(mix(h ^ 0x85EBCA6Bu), 127 - 100, 100 + 21, false);
            const float2 q = div2_rn(make_float2(m, -m), make_float2(dd, dd));
            bad_q += (__float_as_uint(q.x) != __float_as_uint(__fdiv_rn(m, dd))) +
                     (__float_as_uint(q.y) != __float_as_uint(__fdiv_rn(-m, dd)));
            pairs += 2;
        }
    }
    unsigned long long bad_s = 0;
    const uint32_t nv = kEndV - kFirstV;
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < nv; i += gridDim.x * blockDim.x) {
        const float v = __uint_as_float(kFirstV + i);
        const float2 r = sqrt2_rn(make_float2(v, v));
        bad_s += __float_as_uint(r.x) != __float_as_uint(__fsqrt_rn(v));
    }
    // relative errors of the approximate square root (every normal v) and
    // reciprocal (every normal d with a normal reciprocal), in double: the
    // products below are exact in double, the square root correctly rounded
    float err_s = 0.0f, err_r = 0.0f;
    const uint32_t na = kEndV - kFirstNormal;
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < na; i += gridDim.x * blockDim.x) {
        const float v = __uint_as_float(kFirstNormal + i);
        const double s = static_cast<double>(sqrt_approx(v));
        err_s = fmaxf(err_s, static_cast<float>(fabs(s / sqrt(static_cast<double>(v)) - 1.0)));
        if (kFirstNormal + i < kEndD) {
            const double y = static_cast<double>(rcp_approx(v));
            err_r = fmaxf(err_r, static_cast<float>(fabs(y * static_cast<double>(v) - 1.0)));
        }
    }
    atomicAdd(&counts[0], bad_y);
    atomicAdd(&counts[2], bad_q);
    atomicAdd(&counts[3], pairs);
    atomicAdd(&counts[4], bad_s);
    // non-negative floats order like their bit patterns
    atomicMax(&counts[6], static_cast<unsigned long long>(__float_as_uint(err_s)));
    atomicMax(&counts[7], static_cast<unsigned long long>(__float_as_uint(err_r)));
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        atomicAdd(&counts[1], static_cast<unsigned long long>(n));
        atomicAdd(&counts[5], static_cast<unsigned long long>(nv));
    }
}

}  // namespace

cudaError_t launch_selftest_sqrt_div(uint64_t* counts, cudaStream_t st)
{
    const cudaError_t e = cudaMemsetAsync(counts, 0, 8 * sizeof(uint64_t), st);
    if (e != cudaSuccess) return e;
    int grid = 0;
    const cudaError_t eg = persistent_grid(reinterpret_cast<const void*>(selftest_kernel), 256, 0, &grid);
    if (eg != cudaSuccess) return eg;
    selftest_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<unsigned long long*>(counts));
    return cudaGetLastError();
}

}  // namespace q8
