/*
 * q8adamw.h -- C ABI of the GB300 (sm_103a) fused 8-bit blockwise AdamW step
 * with stochastic rounding of BF16 parameters, and its BF16-state variant.
 *
 * Sources, by page title and section:
 *  [BW]  "8-bit Optimizers via Block-wise Quantization": innovations list
 *        (dynamic tree quantization, extended to unipolar data) and method
 *        bullets (2048-element blocks normalised by their absmax, binary
 *        search to an 8-bit index, lookup-table dequantization, states
 *        dequantized, updated in 32 bit and requantized in registers).
 *  [SR]  "Stochastic rounding support for 8-bit optimizers": feature request
 *        (stochastic rounding of BF16 parameter updates, no FP32 master
 *        weights) and scoping comment (FP32-state fallback for small tensors,
 *        stream compatibility).
 *  [MOM] "[Feat]: Stochastic rounding of AdamW momentums": state_dtype choice,
 *        fp32 maths with stochastically rounded write-back of the momentums.
 *  [LLM] "Stochastic Rounding for LLM Training: Theory and Practice": TL;DR
 *        (BF16-AdamW-SR; shared randomness across replicas).
 *
 * Conventions for every entry point:
 *  - Pointers named "device" are CUDA device (or managed/host-mapped) memory
 *    owned by the caller; the library never frees or keeps them.  BF16 values
 *    are passed as their 16-bit patterns (uint16_t).
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream).  Nothing synchronises with the host except the
 *    one-time per-device set-up described at q8_prepare_device().
 *  - Return value: Q8_OK (0), or a negative q8_status.  Argument errors are
 *    detected on the host before anything is launched, and leave all buffers
 *    untouched.  Q8_ERR_CUDA reports a launch or set-up failure.  Faults in
 *    kernels that already ran surface at the caller's next synchronisation.
 *    q8_last_error() returns a message for the last failure on the calling
 *    host thread.
 *  - Non-finite gradients or states give unspecified values (never a fault).
 */
#ifndef Q8ADAMW_H
#define Q8ADAMW_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* q8_stream_t;   /* same type as cudaStream_t */

typedef enum {
    Q8_OK = 0,
    Q8_ERR_NULL = -1,    /* a required pointer is NULL                         */
    Q8_ERR_SIZE = -2,    /* a size is negative or beyond a stated limit        */
    Q8_ERR_ALIGN = -3,   /* a pointer breaks the stated alignment              */
    Q8_ERR_ARG = -4,     /* a hyper-parameter or enum is out of range          */
    Q8_ERR_CUDA = -5     /* the CUDA runtime reported an error                 */
} q8_status;

typedef enum { Q8_SIGNED = 0, Q8_UNSIGNED = 1 } q8_kind;

enum {
    Q8_BLOCK = 2048,          /* [BW] method bullets: elements per absmax block */
    Q8_SMALL_NUMEL = 4096,    /* tensors below this are given fp32 state ([SR]) */
    Q8_MAX_STEP = 0x7FFFFFFF  /* the step counter enters Philox as 32 bits      */
};

/*
 * AdamW hyper-parameters and the stochastic-rounding key.
 *   lr >= 0, 0 <= beta1 < 1, 0 <= beta2 < 1, eps >= 0, weight_decay >= 0 (all
 *   finite); 1 <= step <= Q8_MAX_STEP (the 1-based step being taken, used for
 *   bias correction and as the Philox counter word); seed keys Philox; sr = 1
 *   rounds every BF16 write stochastically, sr = 0 rounds to nearest even.
 * The step forms, in double, a_t = lr*sqrt(1-beta2^t)/(1-beta1^t),
 * eps_t = eps*sqrt(1-beta2^t) and decay = 1 - lr*weight_decay, rounds each to
 * float once, and per element computes in fp32, each multiply-add fused
 * (one rounding) and every other operation rounded on its own:
 *   m = fma(beta1, m, (1-beta1)*g);  v = fma(beta2, v, (1-beta2)*(g*g));
 *   p = fma(-a_t, m / (sqrt(v) + eps_t), p*decay)
 * which is textbook AdamW with decoupled weight decay ([LLM] TL;DR).
 * exact = 1 takes the square root and the division correctly rounded
 * everywhere, so that every output is bit-identical with the plain CPU
 * restatement of these formulas.  exact = 0 (the fast mode) lets the full
 * 2048-blocks of the 8-bit and BF16-state kernels take them from the
 * hardware's approximate square root and reciprocal, when eps_t lies in
 * [2^-36, 2^20] and a_t <= 1 (otherwise the step is exact).  Both feed only
 * the parameter update, so codes, absmax and the BF16 m and v are identical
 * in both modes.  A parameter differs only where the approximation moves its
 * BF16 rounding: elements whose update nearly cancels p*decay are recomputed
 * exactly, so a step's parameters are within one ulp of the exact step's,
 * and about one in a million differs.
 * Any other value of sr or exact is an argument error.
 */
typedef struct {
    double lr, beta1, beta2, eps, weight_decay;
    int64_t step;
    uint64_t seed;
    int32_t sr;
    int32_t exact;
} q8_adamw_hparams;

/*
 * One parameter tensor for adamw8bit_sr_step.  All pointers are device
 * pointers to contiguous 1-D arrays of `numel` elements, 16-byte aligned.
 *   param          bf16, read and written in place
 *   grad           bf16, read only
 *   philox_offset  global Philox index of element 0; a negative value means
 *                  "the sum of numel over the tensors before this one in the
 *                  list" (so one list behaves like one flat tensor)
 * The state an entry carries picks its path:
 * 8-bit state ([BW]; m_codes != NULL): m_codes, v_codes are uint8 indices into
 *   the signed / unsigned codebooks; m_absmax, v_absmax hold one float per
 *   2048-element block (ceil(numel/2048) entries, 4-byte aligned).  m32/v32
 *   must be NULL.  An all-zero state (codes anything, absmax 0) is the fresh
 *   state; canonical zero codes are 127 (m) and 0 (v).  Tensors of 4096 or
 *   more elements are created with this state; a block-aligned slice of one
 *   (element offset a multiple of 2048, its absmax pointers advanced to match,
 *   philox_offset set to the global index of its first element) may be
 *   shorter and stays on this path.
 * fp32 state ([SR] scoping comment: small tensors; m_codes == NULL): m32, v32
 *   are float arrays of numel elements, updated in place; numel < 4096.
 * numel == 0 entries are skipped.
 * Speed only: when the param and grad arrays of every entry of a launch are
 * 32-byte aligned (as PyTorch allocations are), the kernels move them in
 * 32-byte accesses; otherwise in 16-byte ones.  The results are the same.
 * This holds for the one-state steps (momentum8bit_sr_step, lion8bit_sr_step)
 * as well.
 */
typedef struct {
    uint16_t* param;
    const uint16_t* grad;
    int64_t numel;
    int64_t philox_offset;
    uint8_t* m_codes;
    uint8_t* v_codes;
    float* m_absmax;
    float* v_absmax;
    float* m32;
    float* v32;
} q8_tensor8;

/* One tensor for adamw_bf16_sr_step: param, grad, m, v are bf16 device
 * arrays of numel elements (16-byte aligned), param/m/v updated in place. */
typedef struct {
    uint16_t* param;
    const uint16_t* grad;
    uint16_t* m;
    uint16_t* v;
    int64_t numel;
    int64_t philox_offset;
} q8_tensor16;

/*
 * The 256-entry codebook of `kind`, ascending, written to the HOST array
 * out[256] ([BW] innovations list: dynamic tree quantization, signed and
 * unipolar).  Entry j = 0..2^f-1 of decade e is 10^-e*(0.1 + 0.9*(j+1)/2^f)
 * rounded to float; signed: decades e = 0..6 with f = 6-e, mirrored, zero at
 * index 127 and a never-produced duplicate 1.0 at index 255; unsigned:
 * e = 0..7 with f = 7-e, zero at index 0.  Host only; no GPU needed.
 */
int q8_codebook_init(int kind, float* out);

/*
 * Blockwise quantization of n floats ([BW] method bullets): for each
 * 2048-element block (the last may be partial) absmax[b] = max |x|; each x is
 * scaled by the correctly rounded reciprocal of absmax[b], clamped to [-1, 1]
 * and coded as the number of codebook midpoints strictly below it; an
 * all-zero block gets the zero code.  x: device float[n] (16-byte aligned);
 * codes: device uint8[n] (16-byte aligned); absmax: device float[ceil(n/2048)]
 * (4-byte aligned).  For Q8_UNSIGNED, negative x code to 0.  0 <= n < 2^40.
 */
int q8_blockwise_quantize(const float* x, uint8_t* codes, float* absmax, int64_t n,
                          int kind, q8_stream_t stream);

/*
 * Blockwise dequantization ([BW] method bullets): x[i] = C[codes[i]] *
 * absmax[i/2048] with C the codebook of `kind`.  Same layouts as above.
 */
int q8_blockwise_dequantize(const uint8_t* codes, const float* absmax, float* x, int64_t n,
                            int kind, q8_stream_t stream);

/*
 * Fused 8-bit blockwise AdamW step with stochastic rounding of the BF16
 * parameters ([BW] method bullets; [SR] feature request), over a list of
 * `ntensors` tensors (host array).  Per 2048-element block: dequantize m, v,
 * run the AdamW update above in fp32, take the new block absmax of m and v,
 * requantize them, and write p rounded to bf16 with the 16-bit Philox draw of
 * element E = philox_offset + i on stream 0 (see q8_philox_fill).  Entries
 * with fp32 state take the fp32-state path with the same maths.  Blocks
 * never straddle entries.  0 <= ntensors; the list may mix both paths.
 */
int adamw8bit_sr_step(const q8_tensor8* list, int ntensors, const q8_adamw_hparams* hp,
                      q8_stream_t stream);

/*
 * BF16-state AdamW with stochastic rounding ([LLM] BF16-AdamW-SR; [MOM] fp32
 * maths, stochastically rounded write-back of the momentums): m, v are read
 * from bf16, the same fp32 update runs, and p, m, v are written back rounded
 * with Philox streams 0, 1 and 2 respectively.
 */
int adamw_bf16_sr_step(const q8_tensor16* list, int ntensors, const q8_adamw_hparams* hp,
                       q8_stream_t stream);

/*
 * One-state optimizers with a signed 8-bit blockwise first moment and the
 * same stochastically rounded BF16 parameter write ([BW] introduction: Adam
 * and Momentum states; [SR] motivation: 8-bit Lion).  Each x*y + z is one
 * fused fp32 multiply-add; scalars are rounded once to float.
 *   SGD with momentum (PyTorch's definition: dampening 0, weight decay added
 *   to the gradient): d = fma(wd, p, g); m = fma(momentum, m, d);
 *   p = fma(-lr, m, p).
 *   Lion (Chen et al. 2023, "Symbolic Discovery of Optimization Algorithms",
 *   decoupled decay): c = fma(beta1, m, (1-beta1)*g); u = sign(c) (0 at 0);
 *   p = fma(-lr, u, p*(1 - lr*wd)); m = fma(beta2, m, (1-beta2)*g).
 * Hyper-parameters: lr, weight_decay >= 0 and finite; momentum, beta1, beta2
 * in [0, 1); 1 <= step <= Q8_MAX_STEP (the Philox counter word); seed; sr.
 * Tensor list: q8_tensor8 entries with m_codes + m_absmax (8-bit state; any
 * length, block-aligned slices allowed) or m32 (fp32 state, numel < 4096);
 * v_codes, v_absmax and v32 must be NULL.  The parameter draw of element E is
 * r16(E) on Philox stream 0, as for adamw8bit_sr_step.
 */
typedef struct {
    double lr, momentum, weight_decay;
    int64_t step;
    uint64_t seed;
    int32_t sr;
} q8_momentum_hparams;

typedef struct {
    double lr, beta1, beta2, weight_decay;
    int64_t step;
    uint64_t seed;
    int32_t sr;
} q8_lion_hparams;

int momentum8bit_sr_step(const q8_tensor8* list, int ntensors, const q8_momentum_hparams* hp,
                         q8_stream_t stream);
int lion8bit_sr_step(const q8_tensor8* list, int ntensors, const q8_lion_hparams* hp,
                     q8_stream_t stream);

/*
 * The 16-bit random draws the steps use, for inspection: out[i] = r16(E) for
 * E = offset + i, where Philox4x32-10 (Salmon et al., SC'11) with key
 * (seed & 0xffffffff, seed >> 32) and counter (lo32(E/8), stream_id, step,
 * hi32(E/8)) yields four words and element E takes the (E & 1) half (0 = low
 * 16 bits) of word (E >> 1) & 3.  out: device uint16[n] (2-byte aligned).
 */
int q8_philox_fill(uint64_t seed, uint32_t step, uint32_t stream_id, uint64_t offset,
                   int64_t n, uint16_t* out, q8_stream_t stream);

/*
 * Self-test of the packed square root and division the AdamW steps use where
 * they are exact, run on the device against CUDA's IEEE operations.  The
 * division is Markstein's correction (IBM J. Res. Dev. 34(1), 1990) with
 * y = RN(1/d) from the approximate reciprocal and one Newton-Raphson step;
 * the square root is the approximate reciprocal square root with one
 * Newton-Raphson (Heron) correction.
 *   counts[0] = d values whose y differs from __frcp_rn(d), over every
 *               positive normal d with a normal reciprocal (counts[1] of them);
 *   counts[2] = pairs (m, d) whose quotient differs from __fdiv_rn(m, d), over
 *               counts[3] seeded pseudo-random pairs spanning the bounds inside
 *               which the steps use it (2^-90 <= |m| <= 2^26,
 *               2^-100 <= d <= 2^21), both signs of m;
 *   counts[4] = v values whose square root differs from __fsqrt_rn(v), over
 *               every normal v >= 2^-100 (counts[5] of them);
 *   counts[6] = the largest relative error of the approximate square root of
 *               the fast mode (sqrt.approx.ftz.f32) over every normal v, and
 *   counts[7] = that of its approximate reciprocal (rcp.approx.ftz.f32) over
 *               every normal d with a normal reciprocal, each the bit pattern
 *               of a float (errors measured in double precision).
 * counts: device uint64[8] (8-byte aligned), overwritten.  Takes a few
 * seconds on one GPU.
 */
int q8_selftest_sqrt_div(uint64_t* counts, q8_stream_t stream);

/*
 * One-time set-up of the current device: uploads the codebooks and search
 * tables and waits for the copy (a device-wide synchronisation), then works
 * out and caches the launch configuration of every kernel of the library on
 * this device.  Every other entry point does the part it needs on first use;
 * call this yourself before capturing a CUDA graph or when the first step
 * must not synchronise.
 */
int q8_prepare_device(void);

/* Message for the last failure on this host thread ("" if none). */
const char* q8_last_error(void);

/* ABI version: bumped on any change of a signature or struct. */
int q8_abi_version(void);   /* 5 */

#ifdef __cplusplus
}
#endif

#endif /* Q8ADAMW_H */
