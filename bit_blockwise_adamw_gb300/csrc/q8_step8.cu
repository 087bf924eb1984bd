// q8_step8.cu -- the fused 8-bit blockwise AdamW + stochastic-rounding step
// ("8-bit Optimizers via Block-wise Quantization", method bullets: states are
// dequantized, updated in 32 bit and requantized in registers; "Stochastic
// rounding support for 8-bit optimizers", feature request: BF16 parameters
// written with stochastic rounding), and its fp32-state path for tensors below
// 4096 elements (same page, scoping comment).
//
// Layout: one persistent CTA per SM, made of seven independent groups of 128
// threads.  The CTA stages the search tables and a lane-replicated copy of the
// two codebooks in shared memory once (one copy per SM serves all seven
// groups); each group then walks its own contiguous range of 2048-element
// blocks, synchronising only with itself (a named barrier per group).  The
// partial last block of a tensor (if its length is not a multiple of 2048)
// goes to a small second kernel, so the hot loop has only full-block code.
// Per block each of a group's 128 threads owns sixteen contiguous elements:
// streaming loads of grad and param (32 bytes each when the launch's arrays
// allow it, else two 16-byte loads) and of both code arrays.  The kernel is
// bound by instruction issue rather than by DRAM, so the loop is written to
// keep the instruction count down: packed fp32x2 arithmetic (with a packed
// exact square root and division wherever a thread's values allow it, or in
// the fast mode the hardware's approximate ones under a cancellation check),
// codebook lookups whose address is one byte permute and that never share a
// shared-memory bank within a warp, one lookup per code in the search, warp
// reductions with redux.sync.
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

// Each group of 128 threads owns one 2048-element block per iteration,
// sixteen contiguous elements per thread: per-block work (tensor lookup,
// absmax reduction, reciprocals) is spread over twice as many elements as
// with eight, and every code load is a full 16-byte vector.  Seven groups per
// CTA (72 registers a thread); six or eight measured slower.
constexpr int kT8 = 128;
constexpr int kV8 = 16;
constexpr int kW8 = kT8 / 32;
constexpr int kGroups = 7;
static_assert(kT8 * kV8 == kBlock, "one block per group iteration");

// Codebooks replicated per lane: row i (256 bytes) holds Cs[i] for lanes
// 0..31, then Cu[i] for lanes 0..31.  Lane l reads word l of the half-row,
// so the 32 lookups of a warp fall in 32 different banks whatever the codes,
// and the byte offset (code << 8) | (4 * lane) is a single byte permute.
constexpr int kLutBytes = 256 * 256;
constexpr int kRedBytes = 2 * kW8 * 8;                       // per group
constexpr int kSmemBytes = kLutBytes + static_cast<int>(sizeof(DevTables)) + kGroups * kRedBytes;
constexpr int kTailSmemBytes = static_cast<int>(sizeof(DevTables)) + kRedBytes;
static_assert(kSmemBytes <= 227 * 1024, "shared memory of one CTA");

struct Frag {                  // one thread's sixteen elements of one block
    uint32_t g[8], p[8], mc[4], vc[4];
};

// Element-wise loads of a ragged tail (rem < 16 valid elements), zero padded.
// Fully unrolled with predicates so the fragment stays in registers.
__device__ __forceinline__ void load_ragged(const Desc8& d, int64_t i0, int64_t rem, Frag& f)
{
#pragma unroll
    for (int j = 0; j < 8; ++j) { f.g[j] = 0; f.p[j] = 0; }
#pragma unroll
    for (int j = 0; j < 4; ++j) { f.mc[j] = 0x7F7F7F7Fu; f.vc[j] = 0; }
#pragma unroll
    for (int j = 0; j < kV8; ++j) {
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

__device__ __forceinline__ void store_ragged(const Desc8& d, int64_t i0, int64_t rem, const uint32_t po[8],
                                             const uint32_t mo[4], const uint32_t vo[4])
{
#pragma unroll
    for (int j = 0; j < kV8; ++j) {
        if (j < rem) {
            d.p[i0 + j] = static_cast<uint16_t>(po[j >> 1] >> ((j & 1) * 16));   // po: written after the barrier
            d.mq[i0 + j] = static_cast<uint8_t>(mo[j >> 2] >> ((j & 3) * 8));
            d.vq[i0 + j] = static_cast<uint8_t>(vo[j >> 2] >> ((j & 3) * 8));
        }
    }
}

// Prefetch the inputs of local block `lb` into L2: grad, param and both code
// arrays, clipped to whole 16-byte chunks inside the tensor.
__device__ __forceinline__ void prefetch_block(const Desc8& d, int lb)
{
    const int64_t first = static_cast<int64_t>(lb) * kBlock;
    const int64_t n = d.n - first < kBlock ? d.n - first : kBlock;
    const uint32_t b16 = static_cast<uint32_t>(n * 2) & ~15u;
    const uint32_t b8 = static_cast<uint32_t>(n) & ~15u;
    if (b16) {
        prefetch_l2(d.g + first, b16);
        prefetch_l2(d.p + first, b16);
    }
    if (b8) {
        prefetch_l2(d.mq + first, b8);
        prefetch_l2(d.vq + first, b8);
    }
}

__device__ __forceinline__ float absmax4(float2 a, float2 b)
{
    return fmaxf(max3(fabsf(a.x), fabsf(a.y), fabsf(b.x)), fabsf(b.y));
}

// Smallest of four values (min ignores a NaN operand).
__device__ __forceinline__ float min4(float2 a, float2 b)
{
    return fminf(min3(a.x, a.y, b.x), b.y);
}

// Smallest magnitude of four values (min ignores a NaN operand, as max does;
// a NaN m then gives a NaN quotient on either division path).
__device__ __forceinline__ float absmin4(float2 a, float2 b)
{
    return fminf(min3(fabsf(a.x), fabsf(a.y), fabsf(b.x)), fabsf(b.y));
}

// Shared-memory view of the staged tables and of a group's reduction scratch.
struct Smem8 {
    uint32_t lut;              // shared address of the lane-replicated codebooks (main kernel)
    const float* cs;
    const float* cu;
    const uint32_t* cell_s;
    const uint32_t* cell_u;
    uint2* red;                // [2][kW8]
};

// Copy the tables to shared memory at `smem` (all `nthreads` threads of the
// CTA take part, then a CTA barrier).
__device__ __forceinline__ const DevTables* copy_tables(const DevTables* tab, unsigned char* smem, int nthreads)
{
    const uint4* src = reinterpret_cast<const uint4*>(tab);
    uint4* dst = reinterpret_cast<uint4*>(smem);
    for (int i = threadIdx.x; i < static_cast<int>(sizeof(DevTables) / 16); i += nthreads) dst[i] = src[i];
    return reinterpret_cast<const DevTables*>(smem);
}

// The main kernel's shared memory: the lane-replicated codebooks, the tables,
// then one reduction scratch per group.
__device__ __forceinline__ Smem8 stage_main(const DevTables* tab, unsigned char* smem, int grp)
{
    float* lut = reinterpret_cast<float*>(smem);
    for (int i = threadIdx.x; i < kLutBytes / 4; i += kGroups * kT8) {
        const int row = i >> 6, col = i & 63;
        lut[i] = col < 32 ? tab->cs[row] : tab->cu[row];
    }
    const DevTables* t = copy_tables(tab, smem + kLutBytes, kGroups * kT8);
    __syncthreads();
    uint2* red = reinterpret_cast<uint2*>(smem + kLutBytes + sizeof(DevTables) + grp * kRedBytes);
    return Smem8{static_cast<uint32_t>(__cvta_generic_to_shared(smem)), t->cs, t->cu, t->cell_s, t->cell_u, red};
}

// The tail kernel's: the tables and one reduction scratch.
__device__ __forceinline__ Smem8 stage_tail(const DevTables* tab, unsigned char* smem)
{
    const DevTables* t = copy_tables(tab, smem, kT8);
    __syncthreads();
    return Smem8{0u, t->cs, t->cu, t->cell_s, t->cell_u, reinterpret_cast<uint2*>(smem + sizeof(DevTables))};
}

__device__ __forceinline__ float lds_f32(uint32_t addr)
{
    float v;
    asm("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}

// Barrier of one group's 128 threads (id 0 is the whole-CTA barrier, which a
// 128-thread CTA also uses this way).
__device__ __forceinline__ void bar_group(int id)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "n"(kT8) : "memory");
}

// The L2 prefetch the leader thread issues during a block: the inputs of global block
// `target` (when `on`), which lies in the current tensor if target < next.
struct Prefetch {
    const Step8Args* a;
    int target, next, base, ti;
    bool on;
};

// One 2048-element block of one tensor, by one group (`tid` = thread of the
// group, `bar` = the group's barrier id, `lead` = the thread that issues the
// L2 prefetch and stores the block absmax).  FULL: every thread owns sixteen
// valid elements (the hot path: vector loads and stores only, lane-replicated
// codebooks); otherwise the block is the partial last block of its tensor.
// W32: grad and param move in 32-byte accesses (all 32-byte aligned).
// APPROX (full blocks only): the fast mode; the parameter update takes the
// approximate square root and reciprocal (ratio2_approx) instead of the exact
// ones, with its element-by-element cancellation check.
// `it` picks the half of the double-buffered reduction scratch.
// 32-byte streaming load and store (sixteen bf16 values), for launches whose
// grad and param arrays are all 32-byte aligned: one instruction where two
// 16-byte ones were (0.5 % faster at GPT-Neo 6.7B).
__device__ __forceinline__ void ld32(const void* p, uint32_t (&w)[8])
{
    asm volatile("ld.global.cs.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
                 : "l"(p));
}
__device__ __forceinline__ void st32(void* p, const uint32_t (&w)[8])
{
    asm volatile("st.global.cs.v8.u32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                 ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

// The IEEE parameter update of one pair, fma(-a_t, m / (sqrt(v) + eps_t),
// p*decay) with every operation correctly rounded: the rare fallback of both
// modes (the fast mode's cancellation check, the exact mode's range guard),
// kept out of line so that the hot loop's code stays small (0.5 % faster in
// the fast mode, 0.6 % in the bit-exact one, than inlined copies).
__device__ __noinline__ float2 param2_ieee(float eps_t, float nstep, float decay, uint32_t pw, float2 m, float2 v)
{
    const float2 p = bf16x2(pw);
    const float dx = __fadd_rn(__fsqrt_rn(v.x), eps_t), dy = __fadd_rn(__fsqrt_rn(v.y), eps_t);
    return make_float2(__fmaf_rn(nstep, __fdiv_rn(m.x, dx), __fmul_rn(p.x, decay)),
                       __fmaf_rn(nstep, __fdiv_rn(m.y, dy), __fmul_rn(p.y, decay)));
}

template <bool SR, bool FULL, bool W32 = false, bool APPROX = false>
__device__ __forceinline__ void block_step(const Scalars& s, const Desc8& d, int lb, int it, const Smem8& sm,
                                           const Prefetch& pf, int tid, int bar, int lead)
{
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int64_t i0 = static_cast<int64_t>(lb) * kBlock + tid * kV8;
    const int64_t rem = d.n - i0;                        // elements from i0 to the end
    const float2 Mold = splat(d.ma[lb]);
    const float2 Vold = splat(d.va[lb]);

    Frag f;
    if constexpr (FULL) {
        if constexpr (W32) {
            ld32(d.g + i0, f.g);
            ld32(d.p + i0, f.p);
        } else {
            const uint4 g0 = ld_stream16(d.g + i0), g1 = ld_stream16(d.g + i0 + 8);
            const uint4 p0 = ld_stream16(d.p + i0), p1 = ld_stream16(d.p + i0 + 8);
            f.g[0] = g0.x; f.g[1] = g0.y; f.g[2] = g0.z; f.g[3] = g0.w;
            f.g[4] = g1.x; f.g[5] = g1.y; f.g[6] = g1.z; f.g[7] = g1.w;
            f.p[0] = p0.x; f.p[1] = p0.y; f.p[2] = p0.z; f.p[3] = p0.w;
            f.p[4] = p1.x; f.p[5] = p1.y; f.p[6] = p1.z; f.p[7] = p1.w;
        }
        const uint4 mq = ld_stream16(d.mq + i0);
        const uint4 vq = ld_stream16(d.vq + i0);
        f.mc[0] = mq.x; f.mc[1] = mq.y; f.mc[2] = mq.z; f.mc[3] = mq.w;
        f.vc[0] = vq.x; f.vc[1] = vq.y; f.vc[2] = vq.z; f.vc[3] = vq.w;
        // after this block's own loads are in flight, so that the prefetch's
        // work hides in their latency instead of delaying them
        if (tid == lead && pf.on) {
            if (pf.target < pf.next) {
                prefetch_block(d, pf.target - pf.base);
            } else {
                int tq = pf.ti + 1;
                while (pf.target >= pf.a->blk_start[tq + 1]) ++tq;
                prefetch_block(pf.a->d[tq], pf.target - pf.a->blk_start[tq]);
            }
        }
    } else {
        load_ragged(d, i0, rem > 0 ? rem : 0, f);
    }

    // dequantize and update, two elements at a time
    float2 m[8], v[8];
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
        const uint32_t cw = f.mc[k >> 1], vw = f.vc[k >> 1];
        const uint32_t b0 = (k & 1) * 2;
        if constexpr (FULL) {
            // byte offset (code << 8) | (4 * lane): byte b of the code word
            // into byte 1, byte 0 of lw into byte 0, zeros above
            const uint32_t sm0 = 0x5504u | (b0 << 4), sm1 = 0x5504u | ((b0 + 1) << 4);
            m[k] = __fmul2_rn(make_float2(lds_f32(sm.lut + __byte_perm(cw, lw, sm0)),
                                          lds_f32(sm.lut + __byte_perm(cw, lw, sm1))), Mold);
            v[k] = __fmul2_rn(make_float2(lds_f32(sm.lut + 128u + __byte_perm(vw, lw, sm0)),
                                          lds_f32(sm.lut + 128u + __byte_perm(vw, lw, sm1))), Vold);
        } else {
            m[k] = __fmul2_rn(make_float2(sm.cs[byte_of(cw, b0)], sm.cs[byte_of(cw, b0 + 1)]), Mold);
            v[k] = __fmul2_rn(make_float2(sm.cu[byte_of(vw, b0)], sm.cu[byte_of(vw, b0 + 1)]), Vold);
        }
        moments2(s, bf16x2_fma(f.g[k], s.two16), m[k], v[k]);
    }
    if constexpr (!FULL) {
        // padding elements do not count in the block absmax
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (2 * k >= rem) { m[k].x = 0.0f; v[k].x = 0.0f; }
            if (2 * k + 1 >= rem) { m[k].y = 0.0f; v[k].y = 0.0f; }
        }
    }
    // this thread's share of the block absmax of the new moments; with the
    // smallest |m| it also decides whether the packed division is exact here
    const float lm = fmaxf(fmaxf(absmax4(m[0], m[1]), absmax4(m[2], m[3])),
                           fmaxf(absmax4(m[4], m[5]), absmax4(m[6], m[7])));
    const float lv = fmaxf(fmaxf(absmax4(v[0], v[1]), absmax4(v[2], v[3])),
                           fmaxf(absmax4(v[4], v[5]), absmax4(v[6], v[7])));
    if constexpr (FULL && APPROX) {
        // fast mode: the approximate quotient (ratio2_approx), checked for
        // cancellation element by element, two pairs to a branch; pairs that
        // fail take the IEEE square root and division.  The check is written
        // so that a NaN fails it too, so the pairs that pass hold no NaN and
        // round without the quieting (2.4 % faster)
#pragma unroll
        for (int k0 = 0; k0 < 8; k0 += 2) {
            float2 x[2];
            bool redo = false;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float2 q = ratio2_approx(s, m[k0 + j], v[k0 + j]);
                x[j] = step2(s, bf16x2_fma(f.p[k0 + j], s.two16), q);
                const float2 t = __fmul2_rn(q, splat(s.cancel));
                redo = redo | !(fabsf(x[j].x) >= fabsf(t.x)) | !(fabsf(x[j].y) >= fabsf(t.y));
            }
            if (redo) {
#pragma unroll
                for (int j = 0; j < 2; ++j)
                    po[k0 + j] = round2<SR>(param2_ieee(s.eps_t, -s.step_size, s.decay, f.p[k0 + j], m[k0 + j],
                                                        v[k0 + j]), r[k0 + j]);
            } else {
#pragma unroll
                for (int j = 0; j < 2; ++j) po[k0 + j] = round2_num<SR>(x[j], r[k0 + j]);
            }
        }
    } else {
        bool fast = false;
        if constexpr (FULL) {
            const float lo = fminf(fminf(absmin4(m[0], m[1]), absmin4(m[2], m[3])),
                                   fminf(absmin4(m[4], m[5]), absmin4(m[6], m[7])));
            const float lov = fminf(fminf(min4(v[0], v[1]), min4(v[2], v[3])),
                                    fminf(min4(v[4], v[5]), min4(v[6], v[7])));
            fast = s.fast_div && lo >= kDivMinM && lm <= kDivMaxM && lv <= kDivMaxV && lov >= kSqrtMinV;
        }
        if (fast) {
#pragma unroll
            for (int k = 0; k < 8; ++k)
                po[k] = round2<SR>(step2(s, bf16x2(f.p[k]), ratio2_fast(s, m[k], sqrt2_rn(v[k]))), r[k]);
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k)
                po[k] = round2<SR>(param2_ieee(s.eps_t, -s.step_size, s.decay, f.p[k], m[k], v[k]), r[k]);
        }
    }

    if constexpr (FULL) {
        // the parameters do not wait for the block absmax: store them now
        if constexpr (W32) {
            st32(d.p + i0, po);
        } else {
            st_stream16(d.p + i0, make_uint4(po[0], po[1], po[2], po[3]));
            st_stream16(d.p + i0 + 8, make_uint4(po[4], po[5], po[6], po[7]));
        }
    }
    // non-negative floats order like their bit patterns
    const uint32_t wm = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(lm));
    const uint32_t wv = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(lv));
    uint2* red = sm.red + (it & 1) * kW8;                // double-buffered: one barrier per block
    if (lane == 0) red[warp] = make_uint2(wm, wv);
    bar_group(bar);
    const uint2 t = lane < kW8 ? red[lane] : make_uint2(0u, 0u);
    const float M = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, t.x));
    const float V = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, t.y));

    // requantize against the new absmax: scale by RN(1/absmax), look up.  An
    // all-zero block (absmax 0) needs no branch: 1/0 = inf, 0 * inf = NaN, and
    // the saturating multiply maps NaN to +0, whose codes are the zero codes
    // (127 signed, whatever the sign of m; 0 unsigned).
    uint32_t mo[4], vo[4];
    const float im = recip_rn(M), iv = recip_rn(V);
#pragma unroll
    for (int k = 0; k < 8; k += 2) {
        mo[k >> 1] = signed_codes4(count_signed_scaled(m[k].x, im, sm.cell_s), count_signed_scaled(m[k].y, im, sm.cell_s),
                                   count_signed_scaled(m[k + 1].x, im, sm.cell_s),
                                   count_signed_scaled(m[k + 1].y, im, sm.cell_s), m[k].x, m[k].y, m[k + 1].x,
                                   m[k + 1].y);
        vo[k >> 1] = pack4(code_unsigned_scaled(v[k].x, iv, sm.cell_u), code_unsigned_scaled(v[k].y, iv, sm.cell_u),
                           code_unsigned_scaled(v[k + 1].x, iv, sm.cell_u),
                           code_unsigned_scaled(v[k + 1].y, iv, sm.cell_u));
    }

    if constexpr (FULL) {
        st_stream16(d.mq + i0, make_uint4(mo[0], mo[1], mo[2], mo[3]));
        st_stream16(d.vq + i0, make_uint4(vo[0], vo[1], vo[2], vo[3]));
    } else if (rem > 0) {
        store_ragged(d, i0, rem, po, mo, vo);
    }
    if (tid == lead) {
        d.ma[lb] = M;
        d.va[lb] = V;
    }
}

__device__ __forceinline__ bool is_partial(const Desc8& d, int lb)
{
    return static_cast<int64_t>(lb + 1) * kBlock > d.n;
}

// The hot kernel: every full block of the launch's list.  Partial last blocks
// are left to step8_tail_kernel, so this loop carries no ragged-tail code.
// Each group of each CTA takes a contiguous range of the list's blocks (end to
// end over the tensors).
template <bool SR, bool W32, bool APPROX>
__global__ void __launch_bounds__(kT8 * kGroups, 1) step8_kernel(const __grid_constant__ Step8Args a)
{
    extern __shared__ __align__(16) unsigned char smem[];
    const int grp = threadIdx.x / kT8;
    const int tid = threadIdx.x % kT8;
    const Smem8 sm = stage_main(a.tab, smem, grp);
    const int worker = blockIdx.x * kGroups + grp;
    const int nworkers = gridDim.x * kGroups;

    const int begin = static_cast<int>((static_cast<int64_t>(worker) * a.nblocks) / nworkers);
    const int end = static_cast<int>((static_cast<int64_t>(worker + 1) * a.nblocks) / nworkers);
    int ti = begin < end ? find_tensor(a.blk_start, a.nt, begin) : 0;
    // The leader thread of the group does the group's single-thread work: the
    // L2 prefetch (the inputs of the block two ahead, kept in flight; one or
    // none measured slower, three the same) and the block absmax stores.  The
    // CTA's warp w runs on sub-partition w % 4 of the SM, so the leaders of
    // the seven groups sit in warps of different sub-partitions; with all of
    // them in each group's first warp, one sub-partition carried the extra
    // work and the others waited for it at the group barriers (3.4 % slower).
    const int lead = (grp & 3) * 32;
    constexpr int kAhead = 2;
    if (tid == lead) {
        int tq = ti;
        for (int pg = begin; pg < end && pg < begin + kAhead; ++pg) {
            while (pg >= a.blk_start[tq + 1]) ++tq;
            prefetch_block(a.d[tq], pg - a.blk_start[tq]);
        }
    }
    // Tensor by tensor: the descriptor and the tensor's block range are read
    // once per tensor, not once per block.
    for (int gb = begin, it = 0; gb < end;) {
        while (gb >= a.blk_start[ti + 1]) ++ti;
        const Desc8& d = a.d[ti];
        const int base = a.blk_start[ti];
        const int next = a.blk_start[ti + 1];
        const int full_end = min(min(end, next), base + static_cast<int>(d.n / kBlock));
        for (; gb < full_end; ++gb)
            block_step<SR, true, W32, APPROX>(a.s, d, gb - base, it++, sm, Prefetch{&a, gb + kAhead, next, base, ti, gb + kAhead < end},
                                 tid, 1 + grp, lead);
        gb = min(end, next);                             // a partial last block is the tail kernel's
    }
}

// Partial last blocks: one CTA per tensor of the launch, idle unless the
// tensor's length is not a multiple of 2048.
template <bool SR>
__global__ void __launch_bounds__(kT8) step8_tail_kernel(const __grid_constant__ Step8Args a)
{
    const Desc8& d = a.d[blockIdx.x];
    const int lb = static_cast<int>((d.n - 1) / kBlock);
    if (!is_partial(d, lb)) return;
    extern __shared__ __align__(16) unsigned char smem[];
    const Smem8 sm = stage_tail(a.tab, smem);
    block_step<SR, false>(a.s, d, lb, 0, sm, Prefetch{&a, 0, 0, 0, 0, false}, static_cast<int>(threadIdx.x), 0, 0);
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
    if constexpr (SR) draws8(d.e0 + static_cast<uint64_t>(i0), 0u, s.key, r);
#pragma unroll
    for (int j = 0; j < kVec; j += 2) {
        const uint32_t w = round2<SR>(make_float2(pn[j], pn[j + 1]), r[j >> 1]);
        if (j < rem) d.p[i0 + j] = static_cast<uint16_t>(w);
        if (j + 1 < rem) d.p[i0 + j + 1] = static_cast<uint16_t>(w >> 16);
    }
}

template <bool SR, bool W32, bool APPROX>
cudaError_t launch_step8_t(const Step8Args& a, bool has_partial, cudaStream_t st)
{
    int full = 0, unused = 0;
    cudaError_t e = persistent_grid(reinterpret_cast<const void*>(step8_kernel<SR, W32, APPROX>), kT8 * kGroups,
                                    kSmemBytes, &full);
    if (e != cudaSuccess) return e;
    const int per = (a.nblocks + kGroups - 1) / kGroups;
    const int grid = per < full ? per : full;
    if (grid > 0) step8_kernel<SR, W32, APPROX><<<grid, kT8 * kGroups, kSmemBytes, st>>>(a);
    if (has_partial && a.nt > 0) {
        e = persistent_grid(reinterpret_cast<const void*>(step8_tail_kernel<SR>), kT8, kTailSmemBytes, &unused);
        if (e != cudaSuccess) return e;
        step8_tail_kernel<SR><<<a.nt, kT8, kTailSmemBytes, st>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t prepare_step8()
{
    int g = 0;
    const void* ks[] = {reinterpret_cast<const void*>(step8_kernel<true, true, true>),
                        reinterpret_cast<const void*>(step8_kernel<true, true, false>),
                        reinterpret_cast<const void*>(step8_kernel<true, false, true>),
                        reinterpret_cast<const void*>(step8_kernel<true, false, false>),
                        reinterpret_cast<const void*>(step8_kernel<false, true, true>),
                        reinterpret_cast<const void*>(step8_kernel<false, true, false>),
                        reinterpret_cast<const void*>(step8_kernel<false, false, true>),
                        reinterpret_cast<const void*>(step8_kernel<false, false, false>)};
    const void* ts[] = {reinterpret_cast<const void*>(step8_tail_kernel<true>),
                        reinterpret_cast<const void*>(step8_tail_kernel<false>)};
    for (const void* k : ks) {
        const cudaError_t e = persistent_grid(k, kT8 * kGroups, kSmemBytes, &g);
        if (e != cudaSuccess) return e;
    }
    for (const void* k : ts) {
        const cudaError_t e = persistent_grid(k, kT8, kTailSmemBytes, &g);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_step8(const Step8Args& a, cudaStream_t st)
{
    bool has_partial = false;
    for (int i = 0; i < a.nt; ++i) has_partial = has_partial || (a.d[i].n % kBlock) != 0;
    // 32-byte loads and stores of grad and param need every tensor's grad and
    // param 32-byte aligned (block offsets are multiples of 4096 bytes)
    bool w32 = true;
    for (int i = 0; i < a.nt; ++i)
        w32 = w32 && (reinterpret_cast<uintptr_t>(a.d[i].g) % 32) == 0 && (reinterpret_cast<uintptr_t>(a.d[i].p) % 32) == 0;
    const bool ax = a.s.approx != 0;
    if (a.s.sr) {
        if (w32) return ax ? launch_step8_t<true, true, true>(a, has_partial, st) : launch_step8_t<true, true, false>(a, has_partial, st);
        return ax ? launch_step8_t<true, false, true>(a, has_partial, st) : launch_step8_t<true, false, false>(a, has_partial, st);
    }
    if (w32) return ax ? launch_step8_t<false, true, true>(a, has_partial, st) : launch_step8_t<false, true, false>(a, has_partial, st);
    return ax ? launch_step8_t<false, false, true>(a, has_partial, st) : launch_step8_t<false, false, false>(a, has_partial, st);
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
