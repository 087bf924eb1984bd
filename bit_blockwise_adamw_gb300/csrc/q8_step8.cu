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
// of its 256 threads owns eight contiguous elements: 16 bytes of grad and of
// param, 8 bytes of each code array.
//
// Two ways to fetch a block, chosen by the STAGES template argument:
//   STAGES == 0  plain streaming loads into registers at the top of the block;
//   STAGES >= 2  each thread copies its own slice of the next STAGES-1 blocks
//                into a shared-memory ring with cp.async (one commit group per
//                block) and waits for the oldest group: more bytes in flight
//                without more registers.  A thread only ever reads back the
//                slots it wrote itself, so no barrier guards the ring.
#include <cstdlib>

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

// ---------------------------------------------------------------- cp.async
__device__ __forceinline__ void cp_async16(void* dst, const void* src)
{
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(void* dst, const void* src)
{
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

// ---------------------------------------------------------------- smem layout
constexpr int kTablesBytes = 256 * 4 * 2 + 2 * kCellsSigned * 4 + kCellsUnsigned * 4;
constexpr int kRedBytes = 2 * kWarps * 8;
constexpr int kRingOffset = (kTablesBytes + kRedBytes + 15) / 16 * 16;
struct Slot {                  // one block, all threads: 12 KB
    uint4 g[kThreads];
    uint4 p[kThreads];
    uint2 mq[kThreads];
    uint2 vq[kThreads];
};
constexpr int smem_bytes(int stages) { return kRingOffset + stages * static_cast<int>(sizeof(Slot)); }

struct Frag {                  // one thread's eight elements of one block
    uint32_t g[4], p[4], mc[2], vc[2];
};

__device__ __forceinline__ void load_direct(const Desc8& d, int64_t i0, int64_t rem, Frag& f)
{
    if (rem >= kVec) {
        const uint4 g4 = ld_stream16(d.g + i0);
        const uint4 p4 = ld_stream16(d.p + i0);
        const uint2 m2 = ld_stream8(d.mq + i0);
        const uint2 v2 = ld_stream8(d.vq + i0);
        f.g[0] = g4.x; f.g[1] = g4.y; f.g[2] = g4.z; f.g[3] = g4.w;
        f.p[0] = p4.x; f.p[1] = p4.y; f.p[2] = p4.z; f.p[3] = p4.w;
        f.mc[0] = m2.x; f.mc[1] = m2.y; f.vc[0] = v2.x; f.vc[1] = v2.y;
        return;
    }
    // ragged tail of the tensor: element-wise loads, zero padding
#pragma unroll
    for (int j = 0; j < 4; ++j) { f.g[j] = 0; f.p[j] = 0; }
    f.mc[0] = f.mc[1] = 0x7F7F7F7Fu;
    f.vc[0] = f.vc[1] = 0;
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

template <int STAGES>
__global__ void __launch_bounds__(kThreads, STAGES == 0 ? 4 : 3) step8_kernel(const __grid_constant__ Step8Args a)
{
    extern __shared__ __align__(16) unsigned char smem[];
    float* s_cs = reinterpret_cast<float*>(smem);
    float* s_cu = s_cs + 256;
    uint32_t* s_cell_s = reinterpret_cast<uint32_t*>(s_cu + 256);
    uint32_t* s_cell_u = s_cell_s + 2 * kCellsSigned;
    float2* s_red = reinterpret_cast<float2*>(s_cell_u + kCellsUnsigned);   // [2][kWarps]
    Slot* ring = reinterpret_cast<Slot*>(smem + kRingOffset);

    for (int i = threadIdx.x; i < 256; i += kThreads) {
        s_cs[i] = a.tab->cs[i];
        s_cu[i] = a.tab->cu[i];
    }
    for (int i = threadIdx.x; i < 2 * kCellsSigned; i += kThreads) s_cell_s[i] = a.tab->cell_s[i];
    for (int i = threadIdx.x; i < kCellsUnsigned; i += kThreads) s_cell_u[i] = a.tab->cell_u[i];
    __syncthreads();

    const Scalars& s = a.s;
    const bool sr = s.sr != 0;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int begin = static_cast<int>((static_cast<int64_t>(blockIdx.x) * a.nblocks) / gridDim.x);
    const int end = static_cast<int>((static_cast<int64_t>(blockIdx.x + 1) * a.nblocks) / gridDim.x);
    int ti = begin < end ? find_tensor(a.blk_start, a.nt, begin) : 0;

    // prefetch cursor (STAGES >= 2): block `pf` of tensor `tp`
    int pf = begin, tp = ti;
    auto issue = [&](int slot) {
        if (pf < end) {
            while (pf >= a.blk_start[tp + 1]) ++tp;
            const Desc8& d = a.d[tp];
            const int64_t i0 = static_cast<int64_t>(pf - a.blk_start[tp]) * kBlock + tid * kVec;
            if (d.n - i0 >= kVec) {
                Slot& r = ring[slot];
                cp_async16(&r.g[tid], d.g + i0);
                cp_async16(&r.p[tid], d.p + i0);
                cp_async8(&r.mq[tid], d.mq + i0);
                cp_async8(&r.vq[tid], d.vq + i0);
            }
        }
        ++pf;
        cp_async_commit();
    };
    if constexpr (STAGES >= 2) {
#pragma unroll
        for (int k = 0; k < STAGES - 1; ++k) issue(k);
    }

    for (int gb = begin, it = 0; gb < end; ++gb, ++it) {
        while (gb >= a.blk_start[ti + 1]) ++ti;
        const Desc8& d = a.d[ti];
        const int lb = gb - a.blk_start[ti];
        const int64_t i0 = static_cast<int64_t>(lb) * kBlock + tid * kVec;
        const int64_t rem = d.n - i0;                    // elements from i0 to the end
        const float Mold = d.ma[lb];
        const float Vold = d.va[lb];

        Frag f;
        if constexpr (STAGES >= 2) {
            issue((it + STAGES - 1) % STAGES);
            cp_async_wait<STAGES - 1>();
            if (rem >= kVec) {
                const Slot& r = ring[it % STAGES];
                const uint4 g4 = r.g[tid];
                const uint4 p4 = r.p[tid];
                const uint2 m2 = r.mq[tid];
                const uint2 v2 = r.vq[tid];
                f.g[0] = g4.x; f.g[1] = g4.y; f.g[2] = g4.z; f.g[3] = g4.w;
                f.p[0] = p4.x; f.p[1] = p4.y; f.p[2] = p4.z; f.p[3] = p4.w;
                f.mc[0] = m2.x; f.mc[1] = m2.y; f.vc[0] = v2.x; f.vc[1] = v2.y;
            } else {
                load_direct(d, i0, rem, f);
            }
        } else {
            load_direct(d, i0, rem, f);
        }

        // dequantize, update in fp32
        float m[kVec], v[kVec], pn[kVec];
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            const uint32_t cm = (f.mc[j >> 2] >> ((j & 3) * 8)) & 0xFFu;
            const uint32_t cv = (f.vc[j >> 2] >> ((j & 3) * 8)) & 0xFFu;
            m[j] = __fmul_rn(s_cs[cm], Mold);
            v[j] = __fmul_rn(s_cu[cv], Vold);
            const float g = (j & 1) ? bf16hi(f.g[j >> 1]) : bf16lo(f.g[j >> 1]);
            const float p = (j & 1) ? bf16hi(f.p[j >> 1]) : bf16lo(f.p[j >> 1]);
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
        float2* red = s_red + (it & 1) * kWarps;          // double-buffered: one barrier per block
        if (lane == 0) red[warp] = make_float2(lm, lv);
        __syncthreads();
        float M = 0.0f, V = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float2 t = red[w];
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
        if (tid == 0) {
            d.ma[lb] = M;
            d.va[lb] = V;
        }
    }
    if constexpr (STAGES >= 2) cp_async_wait<0>();                 // no copy outlives the CTA
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

template <int STAGES>
cudaError_t launch_step8_t(const Step8Args& a, cudaStream_t st)
{
    static int full = 0;
    const int bytes = smem_bytes(STAGES);
    if (full == 0) {
        const void* k = reinterpret_cast<const void*>(step8_kernel<STAGES>);
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
        full = resident_ctas(k, kThreads, bytes);
        if (full <= 0) return cudaErrorUnknown;
    }
    const int grid = a.nblocks < full ? a.nblocks : full;
    if (grid > 0) step8_kernel<STAGES><<<grid, kThreads, bytes, st>>>(a);
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
    static int variant = -1;
    if (variant < 0) {
        const char* e = std::getenv("Q8_STEP8_STAGES");
        variant = e ? std::atoi(e) : 2;
    }
    switch (variant) {
    case 0: return launch_step8_t<0>(a, st);
    case 3: return launch_step8_t<3>(a, st);
    default: return launch_step8_t<2>(a, st);
    }
}

cudaError_t launch_step32(const Step32Args& a, cudaStream_t st)
{
    if (a.nt > 0) step32_kernel<<<a.nt, kSmallThreads, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace q8
