// q8_step16.cu -- BF16-state AdamW with stochastic rounding ("Stochastic
// Rounding for LLM Training: Theory and Practice", TL;DR: BF16-AdamW-SR;
// "[Feat]: Stochastic rounding of AdamW momentums": fp32 maths with a
// stochastically rounded write-back of both momentums).
//
// Pure streaming: 8 bytes read and 6 written per element.  A persistent grid
// walks contiguous ranges of 2048-element blocks, tensor by tensor: full
// blocks with vector loads and stores only, then the tensor's partial last
// block with per-element bounds.  Each thread owns eight contiguous elements
// and draws three independent Philox streams (p, m, v).
// In the fast mode the full blocks take the approximate square root and
// reciprocal (ratio2_approx) unless the thread's cancellation check fails;
// otherwise, and in the bit-exact mode, the square root and division take the
// packed exact path when all of a thread's eight elements lie inside its
// bounds (q8_device.cuh), the IEEE operations when not.
#include "q8_device.cuh"

namespace q8 {

namespace {

__device__ __forceinline__ int find_tensor16(const int32_t* start, int nt, int gb)
{
    int lo = 0, hi = nt;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (start[mid] <= gb) lo = mid; else hi = mid;
    }
    return lo;
}

__device__ __forceinline__ void load8_bf16(const uint16_t* src, int64_t rem, uint32_t w[4])
{
    if (rem >= kVec) {
        const uint4 q = ld_stream16(src);
        w[0] = q.x; w[1] = q.y; w[2] = q.z; w[3] = q.w;
    } else {
        w[0] = w[1] = w[2] = w[3] = 0;
        for (int j = 0; j < kVec; ++j)
            if (j < rem) w[j >> 1] |= static_cast<uint32_t>(src[j]) << ((j & 1) * 16);
    }
}

__device__ __forceinline__ void store8_bf16(uint16_t* dst, int64_t rem, const uint32_t w[4])
{
    if (rem >= kVec) {
        st_stream16(dst, make_uint4(w[0], w[1], w[2], w[3]));
    } else {
        for (int j = 0; j < kVec; ++j)
            if (j < rem) dst[j] = static_cast<uint16_t>(w[j >> 1] >> ((j & 1) * 16));
    }
}

// One 2048-element block: FULL blocks lie wholly inside the tensor (vector
// loads and stores only); otherwise the partial last block.  APPROX (full
// blocks only): the parameter update takes the approximate square root and
// reciprocal (ratio2_approx); m and v never depend on them.
template <bool SR, bool FULL, bool APPROX = false>
__device__ __forceinline__ void block16(const Scalars& s, const Desc16& d, int lb)
{
    const int64_t i0 = static_cast<int64_t>(lb) * kBlock + threadIdx.x * kVec;
    const int64_t rem = d.n - i0;
    if constexpr (!FULL) {
        if (rem <= 0) return;
    }
    uint32_t gw[4], pw[4], mw[4], vw[4];
    if constexpr (FULL) {
        const uint4 g4 = ld_stream16(d.g + i0), p4 = ld_stream16(d.p + i0);
        const uint4 m4 = ld_stream16(d.m + i0), v4 = ld_stream16(d.v + i0);
        gw[0] = g4.x; gw[1] = g4.y; gw[2] = g4.z; gw[3] = g4.w;
        pw[0] = p4.x; pw[1] = p4.y; pw[2] = p4.z; pw[3] = p4.w;
        mw[0] = m4.x; mw[1] = m4.y; mw[2] = m4.z; mw[3] = m4.w;
        vw[0] = v4.x; vw[1] = v4.y; vw[2] = v4.z; vw[3] = v4.w;
    } else {
        load8_bf16(d.g + i0, rem, gw);
        load8_bf16(d.p + i0, rem, pw);
        load8_bf16(d.m + i0, rem, mw);
        load8_bf16(d.v + i0, rem, vw);
    }

    const uint64_t E = d.e0 + static_cast<uint64_t>(i0);
    uint32_t rp[4] = {0, 0, 0, 0}, rm[4] = {0, 0, 0, 0}, rv[4] = {0, 0, 0, 0};
    if constexpr (SR) {
        draws8(E, 0u, s.key, rp);
        draws8(E, 1u, s.key, rm);
        draws8(E, 2u, s.key, rv);
    }
    uint32_t po[4], mo[4], vo[4];
    float2 m[4], v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        m[k] = bf16x2(mw[k]);
        v[k] = bf16x2(vw[k]);
        moments2(s, bf16x2(gw[k]), m[k], v[k]);
    }
    // fast mode: the approximate quotient with the thread's cancellation
    // check (ratio2_approx); otherwise, or to redo the thread, the packed
    // square root and division where they are exact (bounds in
    // q8_device.cuh); padding elements of a ragged tail are zero and send
    // that thread to the IEEE path
    bool redo = true;
    if constexpr (FULL && APPROX) {
        float qmax = 0.0f, pmin = __uint_as_float(0x7F800000u);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 q = ratio2_approx(s, m[k], v[k]);
            const float2 x = step2(s, bf16x2(pw[k]), q);
            qmax = max3(qmax, fabsf(q.x), fabsf(q.y));
            pmin = min3(pmin, fabsf(x.x), fabsf(x.y));
            po[k] = round2<SR>(x, rp[k]);
        }
        redo = pmin < qmax * s.cancel;
    }
    if (redo) {
        const float lo = fminf(min3(fabsf(m[0].x), fabsf(m[0].y), fabsf(m[1].x)),
                               min3(fabsf(m[1].y), fabsf(m[2].x), fminf(fabsf(m[2].y), fminf(fabsf(m[3].x), fabsf(m[3].y)))));
        const float hi = fmaxf(max3(fabsf(m[0].x), fabsf(m[0].y), fabsf(m[1].x)),
                               max3(fabsf(m[1].y), fabsf(m[2].x), fmaxf(fabsf(m[2].y), fmaxf(fabsf(m[3].x), fabsf(m[3].y)))));
        const float vlo = fminf(min3(v[0].x, v[0].y, v[1].x), min3(v[1].y, v[2].x, fminf(v[2].y, fminf(v[3].x, v[3].y))));
        const float vhi = fmaxf(max3(v[0].x, v[0].y, v[1].x), max3(v[1].y, v[2].x, fmaxf(v[2].y, fmaxf(v[3].x, v[3].y))));
        if (s.fast_div && lo >= kDivMinM && hi <= kDivMaxM && vlo >= kSqrtMinV && vhi <= kDivMaxV) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
                po[k] = round2<SR>(step2(s, bf16x2(pw[k]), ratio2_fast(s, m[k], sqrt2_rn(v[k]))), rp[k]);
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 root = make_float2(__fsqrt_rn(v[k].x), __fsqrt_rn(v[k].y));
                po[k] = round2<SR>(param2(s, bf16x2(pw[k]), m[k], root), rp[k]);
            }
        }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        mo[k] = round2<SR>(m[k], rm[k]);
        vo[k] = round2<SR>(v[k], rv[k]);
    }
    if constexpr (FULL) {
        st_stream16(d.p + i0, make_uint4(po[0], po[1], po[2], po[3]));
        st_stream16(d.m + i0, make_uint4(mo[0], mo[1], mo[2], mo[3]));
        st_stream16(d.v + i0, make_uint4(vo[0], vo[1], vo[2], vo[3]));
    } else {
        store8_bf16(d.p + i0, rem, po);
        store8_bf16(d.m + i0, rem, mo);
        store8_bf16(d.v + i0, rem, vo);
    }
}

template <bool SR, bool APPROX>
__global__ void __launch_bounds__(kThreads, 4) step16_kernel(const __grid_constant__ Step16Args a)
{
    const int begin = static_cast<int>((static_cast<int64_t>(blockIdx.x) * a.nblocks) / gridDim.x);
    const int end = static_cast<int>((static_cast<int64_t>(blockIdx.x + 1) * a.nblocks) / gridDim.x);
    int ti = begin < end ? find_tensor16(a.blk_start, a.nt, begin) : 0;
    // tensor by tensor: full blocks first, then the partial last block
    for (int gb = begin; gb < end;) {
        while (gb >= a.blk_start[ti + 1]) ++ti;
        const Desc16& d = a.d[ti];
        const int base = a.blk_start[ti];
        const int stop = min(end, a.blk_start[ti + 1]);
        const int full_end = min(stop, base + static_cast<int>(d.n / kBlock));
        for (; gb < full_end; ++gb) block16<SR, true, APPROX>(a.s, d, gb - base);
        for (; gb < stop; ++gb) block16<SR, false>(a.s, d, gb - base);
    }
}

}  // namespace

cudaError_t prepare_step16()
{
    int g = 0;
    const void* ks[] = {reinterpret_cast<const void*>(step16_kernel<true, true>),
                        reinterpret_cast<const void*>(step16_kernel<true, false>),
                        reinterpret_cast<const void*>(step16_kernel<false, true>),
                        reinterpret_cast<const void*>(step16_kernel<false, false>)};
    for (const void* k : ks) {
        const cudaError_t e = persistent_grid(k, kThreads, 0, &g);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

namespace {

template <bool SR, bool APPROX>
cudaError_t launch16_t(const Step16Args& a, cudaStream_t st)
{
    int full = 0;
    const cudaError_t e = persistent_grid(reinterpret_cast<const void*>(step16_kernel<SR, APPROX>), kThreads, 0, &full);
    if (e != cudaSuccess) return e;
    const int grid = a.nblocks < full ? a.nblocks : full;
    if (grid > 0) step16_kernel<SR, APPROX><<<grid, kThreads, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_step16(const Step16Args& a, cudaStream_t st)
{
    if (a.s.sr) return a.s.approx ? launch16_t<true, true>(a, st) : launch16_t<true, false>(a, st);
    return a.s.approx ? launch16_t<false, true>(a, st) : launch16_t<false, false>(a, st);
}

}  // namespace q8
