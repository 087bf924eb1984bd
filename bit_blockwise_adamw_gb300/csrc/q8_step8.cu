// q8_step8.cu -- the fused 8-bit blockwise AdamW + stochastic-rounding step
// ("8-bit Optimizers via Block-wise Quantization", method bullets: states are
// dequantized, updated in 32 bit and requantized in registers; "Stochastic
// rounding support for 8-bit optimizers", feature request: BF16 parameters
// written with stochastic rounding), and its fp32-state path for tensors below
// 4096 elements (same page, scoping comment).
//
// Layout: a persistent grid of resident CTAs (a multiple of the SM count);
// each CTA stages the codebooks and the cell search tables in shared memory
// once, then walks a contiguous range of 2048-element blocks.  Per block each
// of its 256 threads owns eight contiguous elements: 16-byte streaming loads
// of grad and param, 8-byte loads of each code array.  The kernel is bound by
// instruction issue rather than by DRAM, so the loop is written to keep the
// instruction count down: packed fp32x2 arithmetic, one shared-memory lookup
// per code, warp reductions with redux.sync, uniform branches only.
#include "q8_device.cuh"

namespace q8 {

namespace {

__device__ __forceinline__ int find_tensor(const int32_t* start, int nt, int gb)
{
    int lo = 0, hi = nt;                 // start[lo] <= gb < start[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (start[mid] <= gb) lo = mid; else hi = mid;
    }
    return lo;
}

constexpr int kSmemBytes = static_cast<int>(sizeof(DevTables)) + 2 * kWarps * 8;

struct Frag {                  // one thread's eight elements of one block
    uint32_t g[4], p[4], mc[2], vc[2];
};

// Element-wise loads of a ragged tail (rem < 8 valid elements), zero padded.
// Fully unrolled with predicates so the fragment stays in registers.
__device__ __forceinline__ void load_ragged(const Desc8& d, int64_t i0, int64_t rem, Frag& f)
{
#pragma unroll
    for (int j = 0; j < 4; ++j) { f.g[j] = 0; f.p[j] = 0; }
    f.mc[0] = f.mc[1] = 0x7F7F7F7Fu;
    f.vc[0] = f.vc[1] = 0;
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
        if (j < rem) {
            const uint32_t sh = (j & 1) * 16;
            f.g[j >> 1] |= static_cast<uint32_t>(d.g[i0 + j]) << sh;
            f.p[j >> 1] |= static_cast<uint32_t>(d.p[i0 + j]) << sh;
            const uint32_t bsh = (j & 3) * 8;
            f.mc[j >> 2] = (f.mc[j >> 2] & ~(0xFFu << bsh)) | (static_cast<uint32_t>(d.mq[i0 + j]) << bsh);
            f.vc[j >> 2] = (f.vc[j >> 2] & ~(0xFFu << bsh)) | (static_cast<uint32_t>(d.vq[i0 + j]) << bsh);
        }
    }
}

__device__ __forceinline__ void store_ragged(const Desc8& d, int64_t i0, int64_t rem, const uint32_t po[4],
                                             const uint32_t mo[2], const uint32_t vo[2])
{
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
        if (j < rem) {
            d.p[i0 + j] = static_cast<uint16_t>(po[j >> 1] >> ((j & 1) * 16));
            d.mq[i0 + j] = static_cast<uint8_t>(mo[j >> 2] >> ((j & 3) * 8));
            d.vq[i0 + j] = static_cast<uint8_t>(vo[j >> 2] >> ((j & 3) * 8));
        }
    }
}

template <bool SR>
__global__ void __launch_bounds__(kThreads, 4) step8_kernel(const __grid_constant__ Step8Args a)
{
    extern __shared__ __align__(16) unsigned char smem[];
    const DevTables* tabs = reinterpret_cast<const DevTables*>(smem);
    const float* s_cs = tabs->cs;
    const float* s_cu = tabs->cu;
    const uint32_t* s_cell_s = tabs->cell_s;
    const uint32_t* s_cell_u = tabs->cell_u;
    uint2* s_red = reinterpret_cast<uint2*>(smem + sizeof(DevTables));   // [2][kWarps]

    {
        const uint4* src = reinterpret_cast<const uint4*>(a.tab);
        uint4* dst = reinterpret_cast<uint4*>(smem);
        for (int i = threadIdx.x; i < static_cast<int>(sizeof(DevTables) / 16); i += kThreads) dst[i] = src[i];
    }
    __syncthreads();

    const Scalars& s = a.s;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int begin = static_cast<int>((static_cast<int64_t>(blockIdx.x) * a.nblocks) / gridDim.x);
    const int end = static_cast<int>((static_cast<int64_t>(blockIdx.x + 1) * a.nblocks) / gridDim.x);
    int ti = begin < end ? find_tensor(a.blk_start, a.nt, begin) : 0;

    for (int gb = begin, it = 0; gb < end; ++gb, ++it) {
        while (gb >= a.blk_start[ti + 1]) ++ti;
        const Desc8& d = a.d[ti];
        const int lb = gb - a.blk_start[ti];
        const int64_t i0 = static_cast<int64_t>(lb) * kBlock + tid * kVec;
        const int64_t rem = d.n - i0;                    // elements from i0 to the end
        const bool full = rem >= kVec;
        const float2 Mold = splat(d.ma[lb]);
        const float2 Vold = splat(d.va[lb]);

        Frag f;
        if (full) {
            const uint4 g4 = ld_stream16(d.g + i0);
            const uint4 p4 = ld_stream16(d.p + i0);
            const uint2 m2 = ld_stream8(d.mq + i0);
            const uint2 v2 = ld_stream8(d.vq + i0);
            f.g[0] = g4.x; f.g[1] = g4.y; f.g[2] = g4.z; f.g[3] = g4.w;
            f.p[0] = p4.x; f.p[1] = p4.y; f.p[2] = p4.z; f.p[3] = p4.w;
            f.mc[0] = m2.x; f.mc[1] = m2.y; f.vc[0] = v2.x; f.vc[1] = v2.y;
        } else {
            load_ragged(d, i0, rem > 0 ? rem : 0, f);
        }

        // dequantize and update, two elements at a time
        float2 m[4], v[4];
        uint32_t po[4];
        uint32_t r[4] = {0, 0, 0, 0};
        if constexpr (SR) draws8(d.e0 + static_cast<uint64_t>(i0), 0u, s, r);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t cw = f.mc[k >> 1], vw = f.vc[k >> 1];
            const int b0 = (k & 1) * 2;
            m[k] = __fmul2_rn(make_float2(s_cs[byte_of(cw, b0)], s_cs[byte_of(cw, b0 + 1)]), Mold);
            v[k] = __fmul2_rn(make_float2(s_cu[byte_of(vw, b0)], s_cu[byte_of(vw, b0 + 1)]), Vold);
            const float2 pn = adamw2(s, bf16x2(f.g[k]), bf16x2(f.p[k]), m[k], v[k]);
            po[k] = round2<SR>(pn, r[k]);
        }

        // block absmax of the new moments (padding elements do not count)
        if (!full) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if (2 * k >= rem) { m[k].x = 0.0f; v[k].x = 0.0f; }
                if (2 * k + 1 >= rem) { m[k].y = 0.0f; v[k].y = 0.0f; }
            }
        }
        const float lm = fmaxf(max3(fabsf(m[0].x), fabsf(m[0].y), fabsf(m[1].x)),
                               max3(fabsf(m[1].y), fabsf(m[2].x), max3(fabsf(m[2].y), fabsf(m[3].x), fabsf(m[3].y))));
        const float lv = fmaxf(max3(v[0].x, v[0].y, v[1].x), max3(v[1].y, v[2].x, max3(v[2].y, v[3].x, v[3].y)));
        // non-negative floats order like their bit patterns
        const uint32_t wm = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(lm));
        const uint32_t wv = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(lv));
        uint2* red = s_red + (it & 1) * kWarps;          // double-buffered: one barrier per block
        if (lane == 0) red[warp] = make_uint2(wm, wv);
        __syncthreads();
        const uint2 t = lane < kWarps ? red[lane] : make_uint2(0u, 0u);
        const float M = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, t.x));
        const float V = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, t.y));

        // requantize against the new absmax: scale by RN(1/absmax), look up
        uint32_t mo[2], vo[2];
        if (M > 0.0f) {
            const float2 im = splat(__frcp_rn(M));
            uint32_t q[8];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 x = __fmul2_rn(m[k], im);
                q[2 * k] = code_signed(x.x, s_cell_s);
                q[2 * k + 1] = code_signed(x.y, s_cell_s);
            }
            mo[0] = pack4(q[0], q[1], q[2], q[3]);
            mo[1] = pack4(q[4], q[5], q[6], q[7]);
        } else {
            mo[0] = mo[1] = 0x7F7F7F7Fu;
        }
        if (V > 0.0f) {
            const float2 iv = splat(__frcp_rn(V));
            uint32_t q[8];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 x = __fmul2_rn(v[k], iv);
                q[2 * k] = code_unsigned_nonneg(x.x, s_cell_u);
                q[2 * k + 1] = code_unsigned_nonneg(x.y, s_cell_u);
            }
            vo[0] = pack4(q[0], q[1], q[2], q[3]);
            vo[1] = pack4(q[4], q[5], q[6], q[7]);
        } else {
            vo[0] = vo[1] = 0u;
        }

        if (full) {
            st_stream16(d.p + i0, make_uint4(po[0], po[1], po[2], po[3]));
            st_stream8(d.mq + i0, make_uint2(mo[0], mo[1]));
            st_stream8(d.vq + i0, make_uint2(vo[0], vo[1]));
        } else if (rem > 0) {
            store_ragged(d, i0, rem, po, mo, vo);
        }
        if (tid == 0) {
            d.ma[lb] = M;
            d.va[lb] = V;
        }
    }
}

// fp32-state path: one CTA per tensor (numel < 4096 = 512 threads x 8).
constexpr int kSmallThreads = kSmall / kVec;

template <bool SR>
__global__ void __launch_bounds__(kSmallThreads) step32_kernel(const __grid_constant__ Step32Args a)
{
    const Desc32& d = a.d[blockIdx.x];
    const Scalars& s = a.s;
    const int64_t i0 = static_cast<int64_t>(threadIdx.x) * kVec;
    const int64_t rem = d.n - i0;
    if (rem <= 0) return;
    float pn[kVec];
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
        if (j < rem) {
            float m = d.m[i0 + j], v = d.v[i0 + j];
            const float g = __uint_as_float(static_cast<uint32_t>(d.g[i0 + j]) << 16);
            const float p = __uint_as_float(static_cast<uint32_t>(d.p[i0 + j]) << 16);
            pn[j] = adamw(s, g, p, m, v);
            d.m[i0 + j] = m;
            d.v[i0 + j] = v;
        } else {
            pn[j] = 0.0f;
        }
    }
    uint32_t r[4] = {0, 0, 0, 0};
    if constexpr (SR) draws8(d.e0 + static_cast<uint64_t>(i0), 0u, s, r);
#pragma unroll
    for (int j = 0; j < kVec; j += 2) {
        const uint32_t w = round2<SR>(make_float2(pn[j], pn[j + 1]), r[j >> 1]);
        if (j < rem) d.p[i0 + j] = static_cast<uint16_t>(w);
        if (j + 1 < rem) d.p[i0 + j + 1] = static_cast<uint16_t>(w >> 16);
    }
}

template <bool SR>
cudaError_t launch_step8_t(const Step8Args& a, cudaStream_t st)
{
    static int full = 0;
    if (full == 0) {
        const void* k = reinterpret_cast<const void*>(step8_kernel<SR>);
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        full = resident_ctas(k, kThreads, kSmemBytes);
        if (full <= 0) return cudaErrorUnknown;
    }
    const int grid = a.nblocks < full ? a.nblocks : full;
    if (grid > 0) step8_kernel<SR><<<grid, kThreads, kSmemBytes, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

int resident_ctas(const void* kernel, int threads, size_t smem)
{
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess)
        return 0;
    return sms * (per_sm > 0 ? per_sm : 1);
}

cudaError_t launch_step8(const Step8Args& a, cudaStream_t st)
{
    return a.s.sr ? launch_step8_t<true>(a, st) : launch_step8_t<false>(a, st);
}

cudaError_t launch_step32(const Step32Args& a, cudaStream_t st)
{
    if (a.nt > 0) {
        if (a.s.sr) step32_kernel<true><<<a.nt, kSmallThreads, 0, st>>>(a);
        else step32_kernel<false><<<a.nt, kSmallThreads, 0, st>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace q8
