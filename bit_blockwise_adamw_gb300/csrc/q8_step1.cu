// q8_step1.cu -- one-state optimizers with an 8-bit blockwise first moment
// and the stochastically rounded BF16 parameter write: SGD with momentum
// ("8-bit Optimizers via Block-wise Quantization", introduction: Adam and
// Momentum states; PyTorch's SGD definition: dampening 0, weight decay added
// to the gradient) and Lion ("Stochastic rounding support for 8-bit
// optimizers", motivation: 8-bit Lion; Chen et al. 2023, decoupled decay).
//
// Same layout as the fused AdamW step: one persistent CTA per SM made of
// seven independent groups of 128 threads, one 2048-element block per group
// iteration, sixteen elements per thread, the signed cell table and a
// lane-replicated signed codebook in shared memory (one copy per SM), the
// group leaders spread over the SM's sub-partitions, partial last blocks in a
// tail kernel, tensors below 4096 elements on an fp32-state kernel.
// Traffic: 8 bytes per parameter plus 8 per block (grad 2, param 2+2, code 1+1).
#include "q8_device.cuh"

namespace q8 {

namespace {

constexpr int kT1 = 128;
constexpr int kV1 = 16;
constexpr int kW1 = kT1 / 32;
static_assert(kT1 * kV1 == kBlock, "one block per CTA iteration");

struct Tables1 {               // the part of DevTables this kernel stages
    float cs[256];
    uint32_t cell_s[kCellSEntries];
};
static_assert(sizeof(Tables1) % 16 == 0, "staged 16 bytes at a time");
constexpr int kGroups1 = 7;                    // 72 registers a thread; eight groups spill
// Lane-replicated signed codebook: row c (256 bytes) holds Cs[c] for lanes
// 0..31 in its first 128 bytes, so lane l's lookup reads word l of the row
// (no two lanes of a warp share a bank) at byte offset (c << 8) | (4 * l),
// one byte permute of the code word.  The rows keep the AdamW kernel's
// 256-byte stride so that the same permute forms the address.
constexpr int kLut1 = 256 * 256;
constexpr int kRed1 = 2 * kW1 * 4;
constexpr int kSmem1 = static_cast<int>(sizeof(Tables1)) + kRed1;
constexpr int kSmem1Main = kLut1 + static_cast<int>(sizeof(Tables1)) + kGroups1 * kRed1;

// Prefetch the inputs of local block `lb` (grad, param, codes), clipped to
// whole 16-byte chunks inside the tensor.
__device__ __forceinline__ void prefetch_block1(const Desc8& d, int lb)
{
    const int64_t first = static_cast<int64_t>(lb) * kBlock;
    const int64_t n = d.n - first < kBlock ? d.n - first : kBlock;
    const uint32_t b16 = static_cast<uint32_t>(n * 2) & ~15u;
    const uint32_t b8 = static_cast<uint32_t>(n) & ~15u;
    if (b16) {
        prefetch_l2(d.g + first, b16);
        prefetch_l2(d.p + first, b16);
    }
    if (b8) prefetch_l2(d.mq + first, b8);
}

__device__ __forceinline__ int find_tensor1(const int32_t* start, int nt, int gb)
{
    int lo = 0, hi = nt;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (start[mid] <= gb) lo = mid; else hi = mid;
    }
    return lo;
}

__device__ __forceinline__ const Tables1* stage1(const DevTables* tab, unsigned char* smem, int nthreads = kT1)
{
    Tables1* t = reinterpret_cast<Tables1*>(smem);
    for (int i = threadIdx.x; i < 256; i += nthreads) t->cs[i] = tab->cs[i];
    const uint4* src = reinterpret_cast<const uint4*>(tab->cell_s);
    uint4* dst = reinterpret_cast<uint4*>(t->cell_s);
    for (int i = threadIdx.x; i < kCellSEntries / 4; i += nthreads) dst[i] = src[i];
    __syncthreads();
    return t;
}

__device__ __forceinline__ float lds_f32_1(uint32_t addr)
{
    float v;
    asm("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}

// Barrier of one group's 128 threads (id 0: the 128-thread tail CTA).
__device__ __forceinline__ void bar_group1(int id)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "n"(kT1) : "memory");
}

// sign(c) as a float: +-1 with the sign bit of c, and +0 for +-0 and NaN
// (|c| > 0 is false for both), built from the bits: one compare, one logic
// op and one select instead of two compares and two selects.
__device__ __forceinline__ float sign1(float c)
{
    return fabsf(c) > 0.0f ? __uint_as_float((__float_as_uint(c) & 0x80000000u) | 0x3F800000u) : 0.0f;
}

// sign(c) of a pair on the FMA pipe: for any nonzero c (subnormals included)
// |c * 2^126 * 2^126| >= 1, so two saturating multiplies give 1 for c > 0 and
// for -c > 0; their difference is +-1, and 0 for +-0 and NaN (a saturating
// multiply maps NaN to 0).  Adding +0 turns a -0 difference into +0, the same
// zero sign1 gives.  Three fewer ALU operations than sign1 for three more on
// the FMA pipe, which the one-state kernel has to spare.
__device__ __forceinline__ float sat_mul(float x, float y)
{
    float r;
    asm("mul.rn.sat.f32 %0, %1, %2;" : "=f"(r) : "f"(x), "f"(y));
    return r;
}

__device__ __forceinline__ float2 sign2(float2 c)
{
    const float2 t = __fmul2_rn(c, splat(0x1p126f));
    const float2 pos = make_float2(sat_mul(t.x, 0x1p126f), sat_mul(t.y, 0x1p126f));
    const float2 neg = make_float2(sat_mul(-t.x, 0x1p126f), sat_mul(-t.y, 0x1p126f));
    return __fadd2_rn(__fadd2_rn(pos, neg2(neg)), splat(0.0f));
}

// The element update of a pair (fp32, each x*y + z fused).
template <int OPT>
__device__ __forceinline__ float2 onestate2(const Scalars1& s, float2 g, float2 p, float2& m)
{
    if constexpr (OPT == kMomentum) {
        const float2 d = __ffma2_rn(splat(s.wd), p, g);
        m = __ffma2_rn(splat(s.a), m, d);
        return __ffma2_rn(splat(s.lr_neg), m, p);
    } else {
        const float2 c = __ffma2_rn(splat(s.a), m, __fmul2_rn(splat(s.oma), g));
        const float2 u = sign2(c);
        const float2 pn = __ffma2_rn(splat(s.lr_neg), u, __fmul2_rn(p, splat(s.decay)));
        m = __ffma2_rn(splat(s.b), m, __fmul2_rn(splat(s.omb), g));
        return pn;
    }
}

template <int OPT>
__device__ __forceinline__ float onestate(const Scalars1& s, float g, float p, float& m)
{
    if constexpr (OPT == kMomentum) {
        const float d = __fmaf_rn(s.wd, p, g);
        m = __fmaf_rn(s.a, m, d);
        return __fmaf_rn(s.lr_neg, m, p);
    } else {
        const float c = __fmaf_rn(s.a, m, __fmul_rn(s.oma, g));
        const float u = sign1(c);
        const float pn = __fmaf_rn(s.lr_neg, u, __fmul_rn(p, s.decay));
        m = __fmaf_rn(s.b, m, __fmul_rn(s.omb, g));
        return pn;
    }
}

// One block, by one group (`tid` = thread of the group, `bar` = its barrier
// id, `lead` = the thread that issues the L2 prefetch and stores the absmax,
// `lut` = shared address of the lane-replicated codebook); FULL = sixteen
// valid elements per thread.
// The L2 prefetch the leader thread issues during a block: the inputs of global block
// `target` (when `on`), which lies in the current tensor if target < next.
struct Prefetch1 {
    const Step1Args* a;
    int target, next, base, ti;
    bool on;
};

// 32-byte streaming load and store (sixteen bf16 values), for launches whose
// grad and param arrays are all 32-byte aligned.
__device__ __forceinline__ void ld32_1(const void* p, uint32_t (&w)[8])
{
    asm volatile("ld.global.cs.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
                 : "l"(p));
}
__device__ __forceinline__ void st32_1(void* p, const uint32_t (&w)[8])
{
    asm volatile("st.global.cs.v8.u32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                 ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

template <int OPT, bool SR, bool FULL, bool W32 = false>
__device__ __forceinline__ void block1(const Scalars1& s, const Desc8& d, int lb, int it, const Tables1* tb,
                                       uint32_t* red2, const Prefetch1& pf, int tid, int bar, int lead, uint32_t lut)
{
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int64_t i0 = static_cast<int64_t>(lb) * kBlock + tid * kV1;
    const int64_t rem = d.n - i0;
    const float2 Mold = splat(d.ma[lb]);

    uint32_t gw[8], pw[8], mc[4];
    if constexpr (FULL) {
        if constexpr (W32) {
            ld32_1(d.g + i0, gw);
            ld32_1(d.p + i0, pw);
        } else {
            const uint4 g0 = ld_stream16(d.g + i0), g1 = ld_stream16(d.g + i0 + 8);
            const uint4 p0 = ld_stream16(d.p + i0), p1 = ld_stream16(d.p + i0 + 8);
            gw[0] = g0.x; gw[1] = g0.y; gw[2] = g0.z; gw[3] = g0.w; gw[4] = g1.x; gw[5] = g1.y; gw[6] = g1.z; gw[7] = g1.w;
            pw[0] = p0.x; pw[1] = p0.y; pw[2] = p0.z; pw[3] = p0.w; pw[4] = p1.x; pw[5] = p1.y; pw[6] = p1.z; pw[7] = p1.w;
        }
        const uint4 mq = ld_stream16(d.mq + i0);
        mc[0] = mq.x; mc[1] = mq.y; mc[2] = mq.z; mc[3] = mq.w;
        // after this block's own loads are in flight
        if (tid == lead && pf.on) {
            if (pf.target < pf.next) {
                prefetch_block1(d, pf.target - pf.base);
            } else {
                int tq = pf.ti + 1;
                while (pf.target >= pf.a->blk_start[tq + 1]) ++tq;
                prefetch_block1(pf.a->d[tq], pf.target - pf.a->blk_start[tq]);
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) { gw[j] = 0; pw[j] = 0; }
#pragma unroll
        for (int j = 0; j < 4; ++j) mc[j] = 0x7F7F7F7Fu;
#pragma unroll
        for (int j = 0; j < kV1; ++j) {
            if (j < rem) {
                gw[j >> 1] |= static_cast<uint32_t>(d.g[i0 + j]) << ((j & 1) * 16);
                pw[j >> 1] |= static_cast<uint32_t>(d.p[i0 + j]) << ((j & 1) * 16);
                const uint32_t bsh = (j & 3) * 8;
                mc[j >> 2] = (mc[j >> 2] & ~(0xFFu << bsh)) | (static_cast<uint32_t>(d.mq[i0 + j]) << bsh);
            }
        }
    }

    float2 m[8];
    uint32_t po[8];
    uint32_t r[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if constexpr (SR) {
        const uint64_t E = d.e0 + static_cast<uint64_t>(i0);
        draws8(E, 0u, s.key, r);
        draws8(E + 8, 0u, s.key, r + 4);
    }
    const uint32_t lw = static_cast<uint32_t>(lane) * 4u;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t cw = mc[k >> 1];
        const uint32_t b0 = (k & 1) * 2;
        if constexpr (FULL)
            m[k] = __fmul2_rn(make_float2(lds_f32_1(lut + __byte_perm(cw, lw, 0x5504u | (b0 << 4))),
                                          lds_f32_1(lut + __byte_perm(cw, lw, 0x5504u | ((b0 + 1) << 4)))), Mold);
        else
            m[k] = __fmul2_rn(make_float2(tb->cs[byte_of(cw, b0)], tb->cs[byte_of(cw, b0 + 1)]), Mold);
        po[k] = round2<SR>(onestate2<OPT>(s, bf16x2(gw[k]), bf16x2(pw[k]), m[k]), r[k]);
    }
    if constexpr (FULL) {
        if constexpr (W32) {
            st32_1(d.p + i0, po);
        } else {
            st_stream16(d.p + i0, make_uint4(po[0], po[1], po[2], po[3]));
            st_stream16(d.p + i0 + 8, make_uint4(po[4], po[5], po[6], po[7]));
        }
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (2 * k >= rem) m[k].x = 0.0f;
            if (2 * k + 1 >= rem) m[k].y = 0.0f;
        }
    }

    float lm = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) lm = max3(lm, fabsf(m[k].x), fabsf(m[k].y));
    const uint32_t wm = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(lm));
    uint32_t* red = red2 + (it & 1) * kW1;
    if (lane == 0) red[warp] = wm;
    bar_group1(bar);
    const float M = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, lane < kW1 ? red[lane] : 0u));

    // absmax 0 needs no branch: m * RN(1/0) saturates to +0, the zero code 127
    uint32_t mo[4];
    const float im = recip_rn(M);
#pragma unroll
    for (int k = 0; k < 8; k += 2) {
        mo[k >> 1] = signed_codes4(count_signed_scaled(m[k].x, im, tb->cell_s), count_signed_scaled(m[k].y, im, tb->cell_s),
                                   count_signed_scaled(m[k + 1].x, im, tb->cell_s),
                                   count_signed_scaled(m[k + 1].y, im, tb->cell_s), m[k].x, m[k].y, m[k + 1].x,
                                   m[k + 1].y);
    }
    if constexpr (FULL) {
        st_stream16(d.mq + i0, make_uint4(mo[0], mo[1], mo[2], mo[3]));
    } else {
#pragma unroll
        for (int j = 0; j < kV1; ++j) {
            if (j < rem) {
                d.p[i0 + j] = static_cast<uint16_t>(po[j >> 1] >> ((j & 1) * 16));
                d.mq[i0 + j] = static_cast<uint8_t>(mo[j >> 2] >> ((j & 3) * 8));
            }
        }
    }
    if (tid == lead) d.ma[lb] = M;
}

__device__ __forceinline__ bool partial1(const Desc8& d, int lb)
{
    return static_cast<int64_t>(lb + 1) * kBlock > d.n;
}

template <int OPT, bool SR, bool W32>
__global__ void __launch_bounds__(kT1 * kGroups1, 1) step1_kernel(const __grid_constant__ Step1Args a)
{
    extern __shared__ __align__(16) unsigned char smem[];
    const int grp = threadIdx.x / kT1;
    const int tid = threadIdx.x % kT1;
    {   // the lane-replicated codebook, then the tables
        float* lut = reinterpret_cast<float*>(smem);
        for (int i = threadIdx.x; i < kLut1 / 4; i += kT1 * kGroups1) {
            const int row = i >> 6, col = i & 63;
            lut[i] = col < 32 ? a.tab->cs[row] : 0.0f;
        }
    }
    const Tables1* tb = stage1(a.tab, smem + kLut1, kT1 * kGroups1);
    const uint32_t lut = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    uint32_t* red = reinterpret_cast<uint32_t*>(smem + kLut1 + sizeof(Tables1) + grp * kRed1);
    // the groups' single-thread work in warps of different SM sub-partitions
    // (warp w of the CTA runs on sub-partition w % 4)
    const int lead = (grp & 3) * 32;
    const int worker = blockIdx.x * kGroups1 + grp;
    const int nworkers = gridDim.x * kGroups1;
    const int begin = static_cast<int>((static_cast<int64_t>(worker) * a.nblocks) / nworkers);
    const int end = static_cast<int>((static_cast<int64_t>(worker + 1) * a.nblocks) / nworkers);
    int ti = begin < end ? find_tensor1(a.blk_start, a.nt, begin) : 0;
    // L2 prefetch: the leader keeps the inputs of the next block in flight
    constexpr int kAhead = 1;
    if (tid == lead) {
        int tq = ti;
        for (int pg = begin; pg < end && pg < begin + kAhead; ++pg) {
            while (pg >= a.blk_start[tq + 1]) ++tq;
            prefetch_block1(a.d[tq], pg - a.blk_start[tq]);
        }
    }
    // tensor by tensor: the descriptor and the tensor's block range are read
    // once per tensor; a partial last block is the tail kernel's
    for (int gb = begin, it = 0; gb < end;) {
        while (gb >= a.blk_start[ti + 1]) ++ti;
        const Desc8& d = a.d[ti];
        const int base = a.blk_start[ti];
        const int next = a.blk_start[ti + 1];
        const int full_end = min(min(end, next), base + static_cast<int>(d.n / kBlock));
        for (; gb < full_end; ++gb)
            block1<OPT, SR, true, W32>(a.s, d, gb - base, it++, tb, red, Prefetch1{&a, gb + kAhead, next, base, ti, gb + kAhead < end},
                                  tid, 1 + grp, lead, lut);
        gb = min(end, next);
    }
}

template <int OPT, bool SR>
__global__ void __launch_bounds__(kT1) step1_tail_kernel(const __grid_constant__ Step1Args a)
{
    const Desc8& d = a.d[blockIdx.x];
    const int lb = static_cast<int>((d.n - 1) / kBlock);
    if (!partial1(d, lb)) return;
    extern __shared__ __align__(16) unsigned char smem[];
    const Tables1* tb = stage1(a.tab, smem);
    uint32_t* red = reinterpret_cast<uint32_t*>(smem + sizeof(Tables1));
    block1<OPT, SR, false>(a.s, d, lb, 0, tb, red, Prefetch1{&a, 0, 0, 0, 0, false}, static_cast<int>(threadIdx.x), 0, 0, 0u);
}

// fp32-state path: one CTA per tensor (numel < 4096 = 512 threads x 8).
constexpr int kSmall1 = kSmall / kVec;

template <int OPT, bool SR>
__global__ void __launch_bounds__(kSmall1) step1_32_kernel(const __grid_constant__ Step1_32Args a)
{
    const Desc32& d = a.d[blockIdx.x];
    const Scalars1& s = a.s;
    const int64_t i0 = static_cast<int64_t>(threadIdx.x) * kVec;
    const int64_t rem = d.n - i0;
    if (rem <= 0) return;
    float pn[kVec];
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
        if (j < rem) {
            float m = d.m[i0 + j];
            const float g = __uint_as_float(static_cast<uint32_t>(d.g[i0 + j]) << 16);
            const float p = __uint_as_float(static_cast<uint32_t>(d.p[i0 + j]) << 16);
            pn[j] = onestate<OPT>(s, g, p, m);
            d.m[i0 + j] = m;
        } else {
            pn[j] = 0.0f;
        }
    }
    uint32_t r[4] = {0, 0, 0, 0};
    if constexpr (SR) draws8(d.e0 + static_cast<uint64_t>(i0), 0u, s.key, r);
#pragma unroll
    for (int j = 0; j < kVec; j += 2) {
        const uint32_t w = round2<SR>(make_float2(pn[j], pn[j + 1]), r[j >> 1]);
        if (j < rem) d.p[i0 + j] = static_cast<uint16_t>(w);
        if (j + 1 < rem) d.p[i0 + j + 1] = static_cast<uint16_t>(w >> 16);
    }
}

template <int OPT, bool SR, bool W32>
cudaError_t launch1(const Step1Args& a, bool has_partial, cudaStream_t st)
{
    int full = 0, unused = 0;
    cudaError_t e = persistent_grid(reinterpret_cast<const void*>(step1_kernel<OPT, SR, W32>), kT1 * kGroups1, kSmem1Main, &full);
    if (e != cudaSuccess) return e;
    const int per = (a.nblocks + kGroups1 - 1) / kGroups1;
    const int grid = per < full ? per : full;
    if (grid > 0) step1_kernel<OPT, SR, W32><<<grid, kT1 * kGroups1, kSmem1Main, st>>>(a);
    if (has_partial && a.nt > 0) {
        e = persistent_grid(reinterpret_cast<const void*>(step1_tail_kernel<OPT, SR>), kT1, kSmem1, &unused);
        if (e != cudaSuccess) return e;
        step1_tail_kernel<OPT, SR><<<a.nt, kT1, kSmem1, st>>>(a);
    }
    return cudaGetLastError();
}

template <int OPT>
cudaError_t launch1_32(const Step1_32Args& a, cudaStream_t st)
{
    if (a.nt > 0) {
        if (a.s.sr) step1_32_kernel<OPT, true><<<a.nt, kSmall1, 0, st>>>(a);
        else step1_32_kernel<OPT, false><<<a.nt, kSmall1, 0, st>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t prepare_step1()
{
    int g = 0;
    const void* ks[] = {reinterpret_cast<const void*>(step1_kernel<kMomentum, true, true>),
                        reinterpret_cast<const void*>(step1_kernel<kMomentum, true, false>),
                        reinterpret_cast<const void*>(step1_kernel<kMomentum, false, true>),
                        reinterpret_cast<const void*>(step1_kernel<kMomentum, false, false>),
                        reinterpret_cast<const void*>(step1_kernel<kLion, true, true>),
                        reinterpret_cast<const void*>(step1_kernel<kLion, true, false>),
                        reinterpret_cast<const void*>(step1_kernel<kLion, false, true>),
                        reinterpret_cast<const void*>(step1_kernel<kLion, false, false>)};
    const void* ts[] = {reinterpret_cast<const void*>(step1_tail_kernel<kMomentum, true>),
                        reinterpret_cast<const void*>(step1_tail_kernel<kMomentum, false>),
                        reinterpret_cast<const void*>(step1_tail_kernel<kLion, true>),
                        reinterpret_cast<const void*>(step1_tail_kernel<kLion, false>)};
    for (const void* k : ks) {
        const cudaError_t e = persistent_grid(k, kT1 * kGroups1, kSmem1Main, &g);
        if (e != cudaSuccess) return e;
    }
    for (const void* k : ts) {
        const cudaError_t e = persistent_grid(k, kT1, kSmem1, &g);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_step1(int opt, const Step1Args& a, cudaStream_t st)
{
    bool has_partial = false, w32 = true;
    for (int i = 0; i < a.nt; ++i) {
        has_partial = has_partial || (a.d[i].n % kBlock) != 0;
        w32 = w32 && (reinterpret_cast<uintptr_t>(a.d[i].g) % 32) == 0 && (reinterpret_cast<uintptr_t>(a.d[i].p) % 32) == 0;
    }
    if (opt == kMomentum) {
        if (a.s.sr) return w32 ? launch1<kMomentum, true, true>(a, has_partial, st) : launch1<kMomentum, true, false>(a, has_partial, st);
        return w32 ? launch1<kMomentum, false, true>(a, has_partial, st) : launch1<kMomentum, false, false>(a, has_partial, st);
    }
    if (a.s.sr) return w32 ? launch1<kLion, true, true>(a, has_partial, st) : launch1<kLion, true, false>(a, has_partial, st);
    return w32 ? launch1<kLion, false, true>(a, has_partial, st) : launch1<kLion, false, false>(a, has_partial, st);
}

cudaError_t launch_step1_32(int opt, const Step1_32Args& a, cudaStream_t st)
{
    return opt == kMomentum ? launch1_32<kMomentum>(a, st) : launch1_32<kLion>(a, st);
}

}  // namespace q8
