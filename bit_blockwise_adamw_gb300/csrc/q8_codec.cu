// q8_codec.cu -- standalone blockwise quantize / dequantize ("8-bit Optimizers
// via Block-wise Quantization", method bullets: per-2048-block absmax, divide
// and binary-search to an 8-bit index; lookup table times absmax) and the
// Philox draw dump used to check the random stream.
#include "q8_device.cuh"

namespace q8 {

namespace {

template <int KIND>
__global__ void __launch_bounds__(kThreads) quantize_kernel(const float* __restrict__ x,
                                                            uint8_t* __restrict__ codes,
                                                            float* __restrict__ absmax, int64_t n,
                                                            int64_t nblocks, const DevTables* tab)
{
    constexpr int kCells = KIND == Q8_SIGNED ? kCellSEntries : kCellsUnsigned;
    __shared__ uint32_t s_cell[kCells];
    __shared__ float s_red[2][kWarps];
    const uint32_t* src = KIND == Q8_SIGNED ? tab->cell_s : tab->cell_u;
    for (int i = threadIdx.x; i < kCells; i += kThreads) s_cell[i] = src[i];
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    int it = 0;
    for (int64_t b = blockIdx.x; b < nblocks; b += gridDim.x, ++it) {
        const int64_t i0 = b * kBlock + threadIdx.x * kVec;
        const int64_t rem = n - i0;
        float xv[kVec];
        if (rem >= kVec) {
            const float4 a = __ldcs(reinterpret_cast<const float4*>(x + i0));
            const float4 c = __ldcs(reinterpret_cast<const float4*>(x + i0 + 4));
            xv[0] = a.x; xv[1] = a.y; xv[2] = a.z; xv[3] = a.w;
            xv[4] = c.x; xv[5] = c.y; xv[6] = c.z; xv[7] = c.w;
        } else {
#pragma unroll
            for (int j = 0; j < kVec; ++j) xv[j] = j < rem ? x[i0 + j] : 0.0f;
        }
        float lm = 0.0f;
#pragma unroll
        for (int j = 0; j < kVec; ++j) lm = fmaxf(lm, fabsf(xv[j]));
        lm = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(lm)));   // lm >= 0
        if (lane == 0) s_red[it & 1][warp] = lm;
        __syncthreads();
        float M = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, s_red[it & 1][w]);

        const float inv = M > 0.0f ? __frcp_rn(M) : 0.0f;
        constexpr uint32_t kZero = KIND == Q8_SIGNED ? 127u : 0u;
        uint32_t q[2] = {0, 0};
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            const uint32_t c = M > 0.0f ? (KIND == Q8_SIGNED ? code_signed_scaled(xv[j], inv, s_cell)
                                                             : code_unsigned_scaled(xv[j], inv, s_cell))
                                        : kZero;
            q[j >> 2] |= (c & 0xFFu) << ((j & 3) * 8);
        }
        if (rem >= kVec) {
            st_stream8(codes + i0, make_uint2(q[0], q[1]));
        } else {
            for (int j = 0; j < kVec; ++j)
                if (j < rem) codes[i0 + j] = static_cast<uint8_t>(q[j >> 2] >> ((j & 3) * 8));
        }
        if (threadIdx.x == 0) absmax[b] = M;
    }
}

__global__ void __launch_bounds__(kThreads) dequantize_kernel(const uint8_t* __restrict__ codes,
                                                              const float* __restrict__ absmax,
                                                              float* __restrict__ x, int64_t n,
                                                              const float* __restrict__ book)
{
    __shared__ float s_book[256];
    for (int i = threadIdx.x; i < 256; i += kThreads) s_book[i] = book[i];
    __syncthreads();
    const int64_t groups = (n + kVec - 1) / kVec;
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; g < groups;
         g += static_cast<int64_t>(gridDim.x) * kThreads) {
        const int64_t i0 = g * kVec;
        const int64_t rem = n - i0;
        const float M = absmax[i0 / kBlock];          // eight elements never straddle a block
        if (rem >= kVec) {
            const uint2 c = __ldcs(reinterpret_cast<const uint2*>(codes + i0));
            float y[kVec];
#pragma unroll
            for (int j = 0; j < kVec; ++j) {
                const uint32_t w = j < 4 ? c.x : c.y;
                y[j] = __fmul_rn(s_book[(w >> ((j & 3) * 8)) & 0xFFu], M);
            }
            __stcs(reinterpret_cast<float4*>(x + i0), make_float4(y[0], y[1], y[2], y[3]));
            __stcs(reinterpret_cast<float4*>(x + i0 + 4), make_float4(y[4], y[5], y[6], y[7]));
        } else {
            for (int j = 0; j < rem; ++j) x[i0 + j] = __fmul_rn(s_book[codes[i0 + j]], M);
        }
    }
}

__global__ void __launch_bounds__(kThreads) philox_fill_kernel(const __grid_constant__ PhiloxKey key,
                                                               uint32_t sid, uint64_t offset,
                                                               int64_t n, uint16_t* __restrict__ out)
{
    const uint64_t first = offset & ~uint64_t(7);
    const uint64_t last = offset + static_cast<uint64_t>(n);          // exclusive
    const uint64_t groups = (last - first + 7) / 8;
    for (uint64_t g = static_cast<uint64_t>(blockIdx.x) * kThreads + threadIdx.x; g < groups;
         g += static_cast<uint64_t>(gridDim.x) * kThreads) {
        const uint64_t E = first + 8 * g;
        uint32_t r[4];
        draws8(E, sid, key, r);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint64_t e = E + j;
            if (e >= offset && e < last) out[e - offset] = static_cast<uint16_t>(r[j >> 1] >> ((j & 1) * 16));
        }
    }
}

}  // namespace

cudaError_t prepare_codec()
{
    int g = 0;
    const void* ks[] = {reinterpret_cast<const void*>(quantize_kernel<Q8_SIGNED>),
                        reinterpret_cast<const void*>(quantize_kernel<Q8_UNSIGNED>),
                        reinterpret_cast<const void*>(dequantize_kernel), reinterpret_cast<const void*>(philox_fill_kernel)};
    for (const void* k : ks) {
        const cudaError_t e = persistent_grid(k, kThreads, 0, &g);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_quantize(const float* x, uint8_t* codes, float* absmax, int64_t n, int kind,
                            const DevTables* tab, cudaStream_t st)
{
    const int64_t nb = (n + kBlock - 1) / kBlock;
    if (nb == 0) return cudaSuccess;
    const void* k = kind == Q8_SIGNED ? reinterpret_cast<const void*>(quantize_kernel<Q8_SIGNED>)
                                      : reinterpret_cast<const void*>(quantize_kernel<Q8_UNSIGNED>);
    int full = 0;
    const cudaError_t e = persistent_grid(k, kThreads, 0, &full);
    if (e != cudaSuccess) return e;
    const int grid = static_cast<int>(nb < full ? nb : full);
    if (kind == Q8_SIGNED) quantize_kernel<Q8_SIGNED><<<grid, kThreads, 0, st>>>(x, codes, absmax, n, nb, tab);
    else quantize_kernel<Q8_UNSIGNED><<<grid, kThreads, 0, st>>>(x, codes, absmax, n, nb, tab);
    return cudaGetLastError();
}

cudaError_t launch_dequantize(const uint8_t* codes, const float* absmax, float* x, int64_t n,
                              int kind, const DevTables* tab, cudaStream_t st)
{
    if (n == 0) return cudaSuccess;
    int full = 0;
    const cudaError_t e = persistent_grid(reinterpret_cast<const void*>(dequantize_kernel), kThreads, 0, &full);
    if (e != cudaSuccess) return e;
    const int64_t groups = (n + kVec - 1) / kVec;
    const int64_t want = (groups + kThreads - 1) / kThreads;
    const int grid = static_cast<int>(want < full ? want : full);
    dequantize_kernel<<<grid, kThreads, 0, st>>>(codes, absmax, x, n, kind == Q8_SIGNED ? tab->cs : tab->cu);
    return cudaGetLastError();
}

cudaError_t launch_philox_fill(const PhiloxKey& key, uint32_t stream_id, uint64_t offset, int64_t n,
                               uint16_t* out, cudaStream_t st)
{
    if (n == 0) return cudaSuccess;
    int full = 0;
    const cudaError_t e = persistent_grid(reinterpret_cast<const void*>(philox_fill_kernel), kThreads, 0, &full);
    if (e != cudaSuccess) return e;
    const uint64_t groups = ((offset & 7) + static_cast<uint64_t>(n) + 7) / 8;
    const uint64_t want = (groups + kThreads - 1) / kThreads;
    const int grid = static_cast<int>(want < static_cast<uint64_t>(full) ? want : full);
    philox_fill_kernel<<<grid, kThreads, 0, st>>>(key, stream_id, offset, n, out);
    return cudaGetLastError();
}

PhiloxKey philox_key(uint64_t seed, uint32_t step)
{
    PhiloxKey k{};
    uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
    for (int r = 0; r < 10; ++r) {
        k.kx[r] = k0;
        k.ky[r] = k1;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    k.step = step;
    return k;
}

}  // namespace q8
