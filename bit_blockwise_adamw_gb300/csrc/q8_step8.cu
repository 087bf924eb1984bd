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
// of its 256 threads owns eight contiguous elements: 16-byte loads of grad and
// param, 8-byte loads of both code arrays, all streamed (evict-first).
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

__device__ __forceinline__ void load_tables(const DevTables* tab, float* cs, float* cu,
                                            uint32_t* cell_s, uint32_t* cell_u)
{
    for (int i = threadIdx.x; i < 256; i += kThreads) {
        cs[i] = tab->cs[i];
        cu[i] = tab->cu[i];
    }
    for (int i = threadIdx.x; i < 2 * kCellsSigned; i += kThreads) cell_s[i] = tab->cell_s[i];
    for (int i = threadIdx.x; i < kCellsUnsigned; i += kThreads) cell_u[i] = tab->cell_u[i];
}

__global__ void __launch_bounds__(kThreads, 4) step8_kernel(const __grid_constant__ Step8Args a)
{
    __shared__ float s_cs[256];
    __shared__ float s_cu[256];
    __shared__ uint32_t s_cell_s[2 * kCellsSigned];
    __shared__ uint32_t s_cell_u[kCellsUnsigned];
    __shared__ float2 s_red[2][kWarps];

    load_tables(a.tab, s_cs, s_cu, s_cell_s, s_cell_u);
    __syncthreads();

    const Scalars& s = a.s;
    const bool sr = s.sr != 0;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int begin = static_cast<int>((static_cast<int64_t>(blockIdx.x) * a.nblocks) / gridDim.x);
    const int end = static_cast<int>((static_cast<int64_t>(blockIdx.x + 1) * a.nblocks) / gridDim.x);
    int ti = begin < end ? find_tensor(a.blk_start, a.nt, begin) : 0;

    for (int gb = begin, it = 0; gb < end; ++gb, ++it) {
        while (gb >= a.blk_start[ti + 1]) ++ti;
        const Desc8& d = a.d[ti];
        const int lb = gb - a.blk_start[ti];
        const int64_t i0 = static_cast<int64_t>(lb) * kBlock + threadIdx.x * kVec;
        const int64_t rem = d.n - i0;                    // elements from i0 to the end
        const float Mold = d.ma[lb];
        const float Vold = d.va[lb];

        uint32_t gw[4], pw[4], mc[2], vc[2];
        if (rem >= kVec) {
            const uint4 g4 = ld_stream16(d.g + i0);
            const uint4 p4 = ld_stream16(d.p + i0);
            const uint2 m2 = ld_stream8(d.mq + i0);
            const uint2 v2 = ld_stream8(d.vq + i0);
            gw[0] = g4.x; gw[1] = g4.y; gw[2] = g4.z; gw[3] = g4.w;
            pw[0] = p4.x; pw[1] = p4.y; pw[2] = p4.z; pw[3] = p4.w;
            mc[0] = m2.x; mc[1] = m2.y; vc[0] = v2.x; vc[1] = v2.y;
        } else {
            // ragged tail of the tensor: element-wise loads, zero padding
#pragma unroll
            for (int j = 0; j < 4; ++j) { gw[j] = 0; pw[j] = 0; }
            mc[0] = mc[1] = 0x7F7F7F7Fu;
            vc[0] = vc[1] = 0;
            for (int j = 0; j < kVec; ++j) {
                if (j < rem) {
                    const uint32_t sh = (j & 1) * 16;
                    gw[j >> 1] |= static_cast<uint32_t>(d.g[i0 + j]) << sh;
                    pw[j >> 1] |= static_cast<uint32_t>(d.p[i0 + j]) << sh;
                    const uint32_t bsh = (j & 3) * 8;
                    mc[j >> 2] = (mc[j >> 2] & ~(0xFFu << bsh)) | (static_cast<uint32_t>(d.mq[i0 + j]) << bsh);
                    vc[j >> 2] = (vc[j >> 2] & ~(0xFFu << bsh)) | (static_cast<uint32_t>(d.vq[i0 + j]) << bsh);
                }
            }
        }

        // dequantize, update in fp32
        float m[kVec], v[kVec], pn[kVec];
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            const uint32_t cm = (mc[j >> 2] >> ((j & 3) * 8)) & 0xFFu;
            const uint32_t cv = (vc[j >> 2] >> ((j & 3) * 8)) & 0xFFu;
            m[j] = __fmul_rn(s_cs[cm], Mold);
            v[j] = __fmul_rn(s_cu[cv], Vold);
            const float g = (j & 1) ? bf16hi(gw[j >> 1]) : bf16lo(gw[j >> 1]);
            const float p = (j & 1) ? bf16hi(pw[j >> 1]) : bf16lo(pw[j >> 1]);
            pn[j] = adamw(s, g, p, m[j], v[j]);
        }

        // parameter: round to bf16 with this element's Philox draw, store
        uint32_t r[4] = {0, 0, 0, 0};
        if (sr) draws8(d.e0 + static_cast<uint64_t>(i0), 0u, s, r);
        uint32_t po[4];
        round8(pn, r, sr, po);
        if (rem >= kVec) {
            st_stream16(d.p + i0, make_uint4(po[0], po[1], po[2], po[3]));
        } else {
            for (int j = 0; j < kVec; ++j)
                if (j < rem) d.p[i0 + j] = static_cast<uint16_t>(po[j >> 1] >> ((j & 1) * 16));
        }

        // block absmax of the new moments (padding contributes zero)
        float lm = 0.0f, lv = 0.0f;
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            if (j < rem) {
                lm = fmaxf(lm, fabsf(m[j]));
                lv = fmaxf(lv, fabsf(v[j]));
            }
        }
        lm = warp_max(lm);
        lv = warp_max(lv);
        if (lane == 0) s_red[it & 1][warp] = make_float2(lm, lv);
        __syncthreads();
        float M = 0.0f, V = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float2 t = s_red[it & 1][w];
            M = fmaxf(M, t.x);
            V = fmaxf(V, t.y);
        }

        // requantize against the new absmax: scale by RN(1/absmax), search
        const float im = M > 0.0f ? __frcp_rn(M) : 0.0f;
        const float iv = V > 0.0f ? __frcp_rn(V) : 0.0f;
        uint32_t mo[2] = {0, 0}, vo[2] = {0, 0};
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            const uint32_t qm = M > 0.0f ? code_signed(__fmul_rn(m[j], im), s_cell_s) : 127u;
            const uint32_t qv = V > 0.0f ? code_unsigned(__fmul_rn(v[j], iv), s_cell_u) : 0u;
            mo[j >> 2] |= qm << ((j & 3) * 8);
            vo[j >> 2] |= qv << ((j & 3) * 8);
        }
        if (rem >= kVec) {
            st_stream8(d.mq + i0, make_uint2(mo[0], mo[1]));
            st_stream8(d.vq + i0, make_uint2(vo[0], vo[1]));
        } else {
            for (int j = 0; j < kVec; ++j) {
                if (j < rem) {
                    d.mq[i0 + j] = static_cast<uint8_t>(mo[j >> 2] >> ((j & 3) * 8));
                    d.vq[i0 + j] = static_cast<uint8_t>(vo[j >> 2] >> ((j & 3) * 8));
                }
            }
        }
        if (threadIdx.x == 0) {
            d.ma[lb] = M;
            d.va[lb] = V;
        }
    }
}

// fp32-state path: one CTA per tensor (numel < 4096 = 512 threads x 8).
constexpr int kSmallThreads = kSmall / kVec;

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
    const bool sr = s.sr != 0;
    uint32_t r[4] = {0, 0, 0, 0};
    if (sr) draws8(d.e0 + static_cast<uint64_t>(i0), 0u, s, r);
    uint32_t po[4];
    round8(pn, r, sr, po);
#pragma unroll
    for (int j = 0; j < kVec; ++j)
        if (j < rem) d.p[i0 + j] = static_cast<uint16_t>(po[j >> 1] >> ((j & 1) * 16));
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
    static int full = 0;
    if (full == 0) full = resident_ctas(reinterpret_cast<const void*>(step8_kernel), kThreads, 0);
    if (full <= 0) return cudaErrorUnknown;
    const int grid = a.nblocks < full ? a.nblocks : full;
    if (grid > 0) step8_kernel<<<grid, kThreads, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_step32(const Step32Args& a, cudaStream_t st)
{
    if (a.nt > 0) step32_kernel<<<a.nt, kSmallThreads, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace q8
