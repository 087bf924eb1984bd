/*
 * q8_oracle.c -- plain, slow, single-threaded CPU oracle for the fused
 * 8-bit blockwise AdamW + stochastic-rounding optimizer step.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker, not the product: it is
 * linked and called only by the test suite, by the smoke check and by the
 * CPU-baseline leg of the benchmark.  It shares no code, header, table or
 * constant generator with the CUDA library; each side implements the same
 * reading of the method on its own.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -fPIC -shared -lm
 * (-ffp-contract=off matters: aarch64 GCC contracts a*b+c into an FMA by
 * default, and every float operation below is meant to round on its own).
 *
 * Sources (cited by page title and section):
 *  [BW]  "8-bit Optimizers via Block-wise Quantization" -- innovations list
 *        (dynamic tree quantization extended to unipolar data) and method
 *        bullets (2048-element blocks, absmax normaliser, normalise then
 *        binary search to an 8-bit index, lookup-table dequantization, update
 *        done in 32 bit in registers).
 *  [SR]  "Stochastic rounding support for 8-bit optimizers" -- feature
 *        request (round the BF16 parameter update up or down with a chance
 *        set by the rounding error; no FP32 master weights) and the scoping
 *        comment (FP32-state fallback for small tensors, weight-decay
 *        baseline, accumulated-update tests).
 *  [MOM] "[Feat]: Stochastic rounding of AdamW momentums" -- state_dtype
 *        flag, add/divide of the update done in fp32, fp32 maths with a
 *        stochastically rounded write-back of the momentums.
 *  [LLM] "Stochastic Rounding for LLM Training: Theory and Practice" --
 *        TL;DR and abstract (BF16-AdamW-SR, shared randomness).
 *  Philox4x32-10 follows Salmon, Moraes, Dror and Shaw, "Parallel Random
 *  Numbers: As Easy as 1, 2, 3" (SC'11), section on the Philox family.
 *  The one-state optimizers follow their published definitions: SGD with
 *  momentum as in PyTorch's SGD (dampening 0, weight decay added to the
 *  gradient) and Lion from Chen et al., "Symbolic Discovery of Optimization
 *  Algorithms" (2023), Algorithm 2 (decoupled weight decay).
 *
 * Readings taken where the pages are silent are listed with each function.
 *
 * Parity pins: every function here is pinned by a CPU test against something
 * other than itself (bit-level decode of the dynamic tree, a library binary
 * search, brute-force nearest code, cuRAND's host Philox generator, exact
 * rational arithmetic, closed forms and statistical properties).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define Q8O_BLOCK 2048      /* [BW] method bullets: blocks of 2048 elements   */
#define Q8O_SMALL 4096      /* tensors with fewer elements keep fp32 state     */

enum { Q8O_SIGNED = 0, Q8O_UNSIGNED = 1 };

/* ------------------------------------------------------------------------ */
/* Codebooks.  [BW] innovations list: "dynamic tree quantization", extended  */
/* to unipolar data.  No table is printed on the pages.  Reading taken: the  */
/* dynamic tree spends its bits after the sign on (a) a run of e zero bits   */
/* giving the decade 10^-e, (b) one indicator bit, (c) f fraction bits that  */
/* place the value linearly inside the decade.  A fraction index k in        */
/* [0, 2^f) maps to 10^-e * (0.1 + 0.9*(k+1)/2^f), i.e. to the right end of  */
/* the k-th of 2^f equal sub-intervals of (0.1*10^-e, 10^-e].  The signed    */
/* book has 7 bits after the sign (e = 0..6, f = 6-e: 127 magnitudes, then   */
/* their negatives and zero: 255 values, padded with a second 1.0 that the   */
/* search never returns); the unsigned book reuses the sign bit as data     */
/* (e = 0..7, f = 7-e: 255 magnitudes and zero).  Each value is the IEEE    */
/* double quotient of two exact integers, rounded once to float.  The code  */
/* stored in memory is the index into the ascending table.                  */
/* ------------------------------------------------------------------------ */

static double pow10_int(int e)
{
    double r = 1.0;
    for (int i = 0; i < e; ++i) r *= 10.0;   /* exact for e <= 22 */
    return r;
}

static int decade_magnitudes(int max_e, int total_bits, float* out)
{
    int n = 0;
    for (int e = 0; e <= max_e; ++e) {
        int f = total_bits - 1 - e;           /* bits left after e zeros + indicator */
        double two_f = (double)(1 << f);
        for (int k = 0; k < (1 << f); ++k) {
            double num = two_f + 9.0 * (double)(k + 1);
            double den = 10.0 * two_f * pow10_int(e);
            out[n++] = (float)(num / den);
        }
    }
    return n;
}

static void sort_floats(float* a, int n)
{
    for (int i = 1; i < n; ++i) {
        float x = a[i];
        int j = i - 1;
        while (j >= 0 && a[j] > x) { a[j + 1] = a[j]; --j; }
        a[j + 1] = x;
    }
}

void q8o_codebook(int kind, float out[256])
{
    float mag[256];
    if (kind == Q8O_UNSIGNED) {
        int n = decade_magnitudes(7, 8, mag);          /* 255 magnitudes */
        out[0] = 0.0f;
        for (int i = 0; i < n; ++i) out[1 + i] = mag[i];
        sort_floats(out, 256);
    } else {
        int n = decade_magnitudes(6, 7, mag);          /* 127 magnitudes */
        sort_floats(mag, n);
        for (int i = 0; i < n; ++i) out[126 - i] = -mag[i];
        out[127] = 0.0f;
        for (int i = 0; i < n; ++i) out[128 + i] = mag[i];
        out[255] = 1.0f;                               /* unreachable pad */
    }
}

/* Decision thresholds between neighbouring codes: the midpoint of the two
 * codes, formed in double (exact for these values) and rounded once. */
void q8o_midpoints(int kind, float out[255])
{
    float c[256];
    q8o_codebook(kind, c);
    for (int j = 0; j < 255; ++j)
        out[j] = (float)(((double)c[j] + (double)c[j + 1]) * 0.5);
}

/* Zero code: the index of 0.0 in the table (written when a block is all zero). */
int q8o_zero_code(int kind) { return kind == Q8O_UNSIGNED ? 0 : 127; }

/* ------------------------------------------------------------------------ */
/* Quantization.  [BW] method bullets: divide by the block maximum, then map */
/* to an 8-bit index by binary search.  Readings: the division by the block  */
/* constant M is a multiplication by the correctly rounded reciprocal 1/M,   */
/* clamped to [-1, 1] (the product can pass 1 by an ulp); the index is the   */
/* number of decision thresholds strictly below the normalised value, so a   */
/* value that sits exactly on a threshold takes the lower code.              */
/* ------------------------------------------------------------------------ */

static int bisect_thresholds(const float mid[255], float x)
{
    int lo = 0, hi = 255;                /* answer lies in [lo, hi] */
    while (lo < hi) {
        int probe = (lo + hi) / 2;
        if (x > mid[probe]) lo = probe + 1;
        else hi = probe;
    }
    return lo;
}

int q8o_search(int kind, float x)
{
    float mid[255];
    q8o_midpoints(kind, mid);
    return bisect_thresholds(mid, x);
}

void q8o_search_many(int kind, const float* x, int64_t n, uint8_t* out)
{
    float mid[255];
    q8o_midpoints(kind, mid);
    for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)bisect_thresholds(mid, x[i]);
}

/* Block absmax: the largest |x| over the block's valid elements. */
static float block_absmax(const float* x, int64_t n)
{
    float m = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float a = fabsf(x[i]);
        if (a > m) m = a;
    }
    return m;
}

static void quantize_block(const float mid[255], int zero_code,
                           const float* x, int64_t n, uint8_t* codes, float* absmax)
{
    float M = block_absmax(x, n);
    *absmax = M;
    float inv = M > 0.0f ? 1.0f / M : 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        if (M == 0.0f) { codes[i] = (uint8_t)zero_code; continue; }
        float y = x[i] * inv;
        if (y > 1.0f) y = 1.0f;
        if (y < -1.0f) y = -1.0f;
        codes[i] = (uint8_t)bisect_thresholds(mid, y);
    }
}

void q8o_quantize(int kind, const float* x, int64_t n, uint8_t* codes, float* absmax)
{
    float mid[255];
    q8o_midpoints(kind, mid);
    for (int64_t b = 0; b * Q8O_BLOCK < n; ++b) {
        int64_t len = n - b * Q8O_BLOCK;
        if (len > Q8O_BLOCK) len = Q8O_BLOCK;
        quantize_block(mid, q8o_zero_code(kind), x + b * Q8O_BLOCK, len,
                       codes + b * Q8O_BLOCK, absmax + b);
    }
}

/* [BW] method bullets: look the code up and multiply by the block maximum. */
void q8o_dequantize(int kind, const uint8_t* codes, const float* absmax, int64_t n, float* out)
{
    float c[256];
    q8o_codebook(kind, c);
    for (int64_t i = 0; i < n; ++i) out[i] = c[codes[i]] * absmax[i / Q8O_BLOCK];
}

/* ------------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon et al., SC'11).  One round maps the counter        */
/* (c0,c1,c2,c3) under key (k0,k1) to (hi(M1*c2)^c1^k0, lo(M1*c2),          */
/* hi(M0*c0)^c3^k1, lo(M0*c0)); the key is bumped by the Weyl constants     */
/* between rounds; ten rounds.                                               */
/* Reading for the keying (the pages only ask for shared randomness):       */
/*   key     = (seed & 0xffffffff, seed >> 32)                               */
/*   counter = (low 32 bits of E/8, stream, step, high 32 bits of E/8)       */
/* where E is the global element index.  One call yields 8 random 16-bit    */
/* values: element E takes half (E & 1) (0 = low half) of word (E >> 1) & 3. */
/* Streams: 0 = parameter, 1 = first moment, 2 = second moment.             */
/* ------------------------------------------------------------------------ */

void q8o_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4])
{
    const uint64_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t p0 = M0 * (uint64_t)c0;
        uint64_t p1 = M1 * (uint64_t)c2;
        uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        uint32_t n1 = (uint32_t)p1;
        uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        uint32_t n3 = (uint32_t)p0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        k0 += W0; k1 += W1;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

uint16_t q8o_r16(uint64_t seed, uint32_t step, uint32_t stream, uint64_t E)
{
    uint64_t group = E >> 3;
    uint32_t ctr[4] = { (uint32_t)group, stream, step, (uint32_t)(group >> 32) };
    uint32_t key[2] = { (uint32_t)seed, (uint32_t)(seed >> 32) };
    uint32_t w[4];
    q8o_philox4x32_10(ctr, key, w);
    uint32_t word = w[(E >> 1) & 3];
    return (uint16_t)((E & 1) ? (word >> 16) : (word & 0xFFFFu));
}

void q8o_philox_fill(uint64_t seed, uint32_t step, uint32_t stream,
                     uint64_t offset, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = q8o_r16(seed, step, stream, offset + (uint64_t)i);
}

/* ------------------------------------------------------------------------ */
/* Rounding fp32 -> bf16.  [SR] feature request: round up or down with a    */
/* chance set by the rounding error.  With r uniform on [0, 2^16), adding r */
/* to the fp32 bit pattern and keeping the top 16 bits rounds the magnitude */
/* up exactly when r >= 2^16 - (low 16 bits), i.e. with probability         */
/* low/2^16, which makes the result unbiased.  NaN becomes the quiet NaN    */
/* 0x7FC0.  Round-to-nearest-even is the non-stochastic comparison mode.    */
/* ------------------------------------------------------------------------ */

static uint32_t f32_bits(float x) { uint32_t u; memcpy(&u, &x, 4); return u; }
static float bits_f32(uint32_t u) { float x; memcpy(&x, &u, 4); return x; }

uint16_t q8o_sr_bf16(float x, uint16_t r)
{
    if (isnan(x)) return 0x7FC0u;
    return (uint16_t)((f32_bits(x) + (uint32_t)r) >> 16);
}

uint16_t q8o_rne_bf16(float x)
{
    if (isnan(x)) return 0x7FC0u;
    uint32_t u = f32_bits(x);
    return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

float q8o_bf16_to_f32(uint16_t h) { return bits_f32((uint32_t)h << 16); }

/* ------------------------------------------------------------------------ */
/* AdamW.  [LLM] TL;DR names AdamW; [BW] method bullets: the update runs in */
/* 32 bit; [MOM] the add and divide of the parameter update are fp32;       */
/* [SR] no fp32 master copy of the parameters.  Reading (decoupled weight   */
/* decay on the old parameter, bias correction folded into the step size):  */
/*   m  = b1*m + (1-b1)*g                                                    */
/*   v  = b2*v + (1-b2)*g*g                                                  */
/*   p  = p*(1 - lr*wd) - a_t * m / (sqrt(v) + eps_t)                        */
/*   a_t = lr*sqrt(1-b2^t)/(1-b1^t),  eps_t = eps*sqrt(1-b2^t)               */
/* which is exactly lr*mhat/(sqrt(vhat)+eps) with mhat = m/(1-b1^t) and     */
/* vhat = v/(1-b2^t).  Scalars are formed in double (b^t by libm pow) and   */
/* rounded once to float.  In fp32, each "x*y + z" above is one fused       */
/* multiply-add (fmaf: one rounding), every other operation rounds on its   */
/* own:                                                                      */
/*   m = fma(b1, m, (1-b1)*g)                                                */
/*   v = fma(b2, v, (1-b2)*(g*g))                                            */
/*   p = fma(-a_t, m / (sqrt(v) + eps_t), p*decay)                           */
/* ------------------------------------------------------------------------ */

typedef struct {
    double lr, beta1, beta2, eps, weight_decay;
    int64_t step;
    uint64_t seed;
    int32_t sr;          /* 1 = stochastic rounding, 0 = round to nearest even */
} q8o_hparams;

typedef struct { float b1, omb1, b2, omb2, eps_t, step_size, decay; } q8o_scalars;

void q8o_step_scalars(const q8o_hparams* hp, q8o_scalars* s)
{
    double t = (double)hp->step;
    double bc1 = 1.0 - pow(hp->beta1, t);
    double bc2 = 1.0 - pow(hp->beta2, t);
    double rbc2 = sqrt(bc2);
    s->b1 = (float)hp->beta1;
    s->omb1 = (float)(1.0 - hp->beta1);
    s->b2 = (float)hp->beta2;
    s->omb2 = (float)(1.0 - hp->beta2);
    s->eps_t = (float)(hp->eps * rbc2);
    s->step_size = (float)(hp->lr * rbc2 / bc1);
    s->decay = (float)(1.0 - hp->lr * hp->weight_decay);
}

/* One element: returns the new fp32 parameter, updates *m and *v in place. */
float q8o_adamw_element(const q8o_scalars* s, float g, float p, float* m, float* v)
{
    float mg = s->omb1 * g;
    float mn = fmaf(s->b1, *m, mg);
    float gg = g * g;
    float vg = s->omb2 * gg;
    float vn = fmaf(s->b2, *v, vg);
    float den = sqrtf(vn) + s->eps_t;
    float ratio = mn / den;
    float pd = p * s->decay;
    *m = mn;
    *v = vn;
    return fmaf(-s->step_size, ratio, pd);
}

static uint16_t round_param(const q8o_hparams* hp, float x, uint32_t stream, uint64_t E)
{
    if (!hp->sr) return q8o_rne_bf16(x);
    return q8o_sr_bf16(x, q8o_r16(hp->seed, (uint32_t)hp->step, stream, E));
}

/* ------------------------------------------------------------------------ */
/* Tensor-level steps.                                                       */
/* ------------------------------------------------------------------------ */

typedef struct {
    uint16_t* param;        /* bf16 bits, updated in place                    */
    const uint16_t* grad;   /* bf16 bits                                      */
    int64_t numel;
    int64_t philox_offset;  /* global index of element 0; < 0 = running sum   */
    uint8_t* m_codes;       /* 8-bit path (numel >= 4096)                     */
    uint8_t* v_codes;
    float* m_absmax;        /* one per 2048-element block                     */
    float* v_absmax;
    float* m32;             /* fp32-state path (numel < 4096)                 */
    float* v32;
} q8o_tensor8;

typedef struct {
    uint16_t* param;
    const uint16_t* grad;
    uint16_t* m;            /* bf16 first moment                              */
    uint16_t* v;            /* bf16 second moment                             */
    int64_t numel;
    int64_t philox_offset;
} q8o_tensor16;

/* 8-bit state, one tensor, offset E0 given.  [BW] method bullets: per block,
 * dequantize, update in 32 bit, then requantize against the new absmax. */
void q8o_adamw8bit_tensor(const q8o_tensor8* t, uint64_t E0, const q8o_hparams* hp)
{
    q8o_scalars s;
    q8o_step_scalars(hp, &s);
    float cs[256], cu[256], mid_s[255], mid_u[255];
    q8o_codebook(Q8O_SIGNED, cs);
    q8o_codebook(Q8O_UNSIGNED, cu);
    q8o_midpoints(Q8O_SIGNED, mid_s);
    q8o_midpoints(Q8O_UNSIGNED, mid_u);
    float mb[Q8O_BLOCK], vb[Q8O_BLOCK];
    for (int64_t b = 0; b * Q8O_BLOCK < t->numel; ++b) {
        int64_t base = b * Q8O_BLOCK;
        int64_t len = t->numel - base;
        if (len > Q8O_BLOCK) len = Q8O_BLOCK;
        float Mold = t->m_absmax[b], Vold = t->v_absmax[b];
        for (int64_t i = 0; i < len; ++i) {
            int64_t e = base + i;
            float m = cs[t->m_codes[e]] * Mold;
            float v = cu[t->v_codes[e]] * Vold;
            float g = q8o_bf16_to_f32(t->grad[e]);
            float p = q8o_bf16_to_f32(t->param[e]);
            float pn = q8o_adamw_element(&s, g, p, &m, &v);
            t->param[e] = round_param(hp, pn, 0, E0 + (uint64_t)e);
            mb[i] = m;
            vb[i] = v;
        }
        quantize_block(mid_s, q8o_zero_code(Q8O_SIGNED), mb, len, t->m_codes + base, t->m_absmax + b);
        quantize_block(mid_u, q8o_zero_code(Q8O_UNSIGNED), vb, len, t->v_codes + base, t->v_absmax + b);
    }
}

/* fp32 state, one tensor.  [SR] scoping comment: small tensors keep fp32
 * state; the element maths is the same as on the 8-bit path. */
void q8o_adamw32_tensor(const q8o_tensor8* t, uint64_t E0, const q8o_hparams* hp)
{
    q8o_scalars s;
    q8o_step_scalars(hp, &s);
    for (int64_t e = 0; e < t->numel; ++e) {
        float m = t->m32[e], v = t->v32[e];
        float g = q8o_bf16_to_f32(t->grad[e]);
        float p = q8o_bf16_to_f32(t->param[e]);
        float pn = q8o_adamw_element(&s, g, p, &m, &v);
        t->param[e] = round_param(hp, pn, 0, E0 + (uint64_t)e);
        t->m32[e] = m;
        t->v32[e] = v;
    }
}

/* BF16 state ([LLM] BF16-AdamW-SR; [MOM] fp32 maths, stochastically rounded
 * write-back of both momentums): p, m, v each on its own Philox stream. */
void q8o_adamw_bf16_tensor(const q8o_tensor16* t, uint64_t E0, const q8o_hparams* hp)
{
    q8o_scalars s;
    q8o_step_scalars(hp, &s);
    for (int64_t e = 0; e < t->numel; ++e) {
        float m = q8o_bf16_to_f32(t->m[e]);
        float v = q8o_bf16_to_f32(t->v[e]);
        float g = q8o_bf16_to_f32(t->grad[e]);
        float p = q8o_bf16_to_f32(t->param[e]);
        float pn = q8o_adamw_element(&s, g, p, &m, &v);
        uint64_t E = E0 + (uint64_t)e;
        t->param[e] = round_param(hp, pn, 0, E);
        t->m[e] = round_param(hp, m, 1, E);
        t->v[e] = round_param(hp, v, 2, E);
    }
}

/* Whole list.  [SR] scoping comment: small tensors keep fp32 state.  The
 * 4096-element threshold decides which state a tensor is created with; in a
 * step, each entry takes the path of the state it carries (8-bit when it has
 * codes, fp32 otherwise), so a block-aligned slice of a large tensor stays on
 * the 8-bit path.  A negative philox_offset means the running sum of the
 * numels of the entries before it in list order. */
int q8o_adamw8bit_sr_step(const q8o_tensor8* list, int n, const q8o_hparams* hp)
{
    uint64_t running = 0;
    for (int i = 0; i < n; ++i) {
        const q8o_tensor8* t = &list[i];
        uint64_t E0 = t->philox_offset >= 0 ? (uint64_t)t->philox_offset : running;
        if (t->m_codes) q8o_adamw8bit_tensor(t, E0, hp);
        else q8o_adamw32_tensor(t, E0, hp);
        running += (uint64_t)t->numel;
    }
    return 0;
}

int q8o_adamw_bf16_sr_step(const q8o_tensor16* list, int n, const q8o_hparams* hp)
{
    uint64_t running = 0;
    for (int i = 0; i < n; ++i) {
        const q8o_tensor16* t = &list[i];
        uint64_t E0 = t->philox_offset >= 0 ? (uint64_t)t->philox_offset : running;
        q8o_adamw_bf16_tensor(t, E0, hp);
        running += (uint64_t)t->numel;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* One-state optimizers with an 8-bit blockwise first moment and the same   */
/* SR parameter write.  [BW] introduction: optimizer states of Adam and     */
/* Momentum; [SR] motivation: 8-bit Lion.  fp32, each x*y + z fused:        */
/*   Momentum: d = fma(wd, p, g); m = fma(mu, m, d); p = fma(-lr, m, p)     */
/*   Lion:     c = fma(b1, m, (1-b1)*g); u = sign(c) (0 for c = 0);         */
/*             p = fma(-lr, u, p*(1 - lr*wd)); m = fma(b2, m, (1-b2)*g)     */
/* Hyper-parameters travel in q8o_hparams: momentum uses beta1 as mu; eps   */
/* is unused.                                                               */
/* ------------------------------------------------------------------------ */

enum { Q8O_MOMENTUM = 0, Q8O_LION = 1 };

typedef struct { float lr_neg, a, oma, b, omb, decay, wd; } q8o_scalars1;

void q8o_step_scalars1(int opt, const q8o_hparams* hp, q8o_scalars1* s)
{
    s->lr_neg = (float)(-hp->lr);
    s->a = (float)hp->beta1;
    s->oma = (float)(1.0 - hp->beta1);
    s->b = (float)hp->beta2;
    s->omb = (float)(1.0 - hp->beta2);
    s->decay = (float)(1.0 - hp->lr * hp->weight_decay);
    s->wd = (float)hp->weight_decay;
    (void)opt;
}

/* One element: returns the new fp32 parameter, updates *m in place. */
float q8o_onestate_element(int opt, const q8o_scalars1* s, float g, float p, float* m)
{
    if (opt == Q8O_MOMENTUM) {
        float d = fmaf(s->wd, p, g);
        float mn = fmaf(s->a, *m, d);
        *m = mn;
        return fmaf(s->lr_neg, mn, p);
    }
    float c = fmaf(s->a, *m, s->oma * g);
    float u = c > 0.0f ? 1.0f : (c < 0.0f ? -1.0f : 0.0f);
    float pn = fmaf(s->lr_neg, u, p * s->decay);
    *m = fmaf(s->b, *m, s->omb * g);
    return pn;
}

/* 8-bit state, one tensor (m_codes / m_absmax; the v fields are unused). */
void q8o_onestate8bit_tensor(int opt, const q8o_tensor8* t, uint64_t E0, const q8o_hparams* hp)
{
    q8o_scalars1 s;
    q8o_step_scalars1(opt, hp, &s);
    float cs[256], mid_s[255];
    q8o_codebook(Q8O_SIGNED, cs);
    q8o_midpoints(Q8O_SIGNED, mid_s);
    float mb[Q8O_BLOCK];
    for (int64_t b = 0; b * Q8O_BLOCK < t->numel; ++b) {
        int64_t base = b * Q8O_BLOCK;
        int64_t len = t->numel - base;
        if (len > Q8O_BLOCK) len = Q8O_BLOCK;
        float Mold = t->m_absmax[b];
        for (int64_t i = 0; i < len; ++i) {
            int64_t e = base + i;
            float m = cs[t->m_codes[e]] * Mold;
            float g = q8o_bf16_to_f32(t->grad[e]);
            float p = q8o_bf16_to_f32(t->param[e]);
            float pn = q8o_onestate_element(opt, &s, g, p, &m);
            t->param[e] = round_param(hp, pn, 0, E0 + (uint64_t)e);
            mb[i] = m;
        }
        quantize_block(mid_s, q8o_zero_code(Q8O_SIGNED), mb, len, t->m_codes + base, t->m_absmax + b);
    }
}

void q8o_onestate32_tensor(int opt, const q8o_tensor8* t, uint64_t E0, const q8o_hparams* hp)
{
    q8o_scalars1 s;
    q8o_step_scalars1(opt, hp, &s);
    for (int64_t e = 0; e < t->numel; ++e) {
        float m = t->m32[e];
        float g = q8o_bf16_to_f32(t->grad[e]);
        float p = q8o_bf16_to_f32(t->param[e]);
        float pn = q8o_onestate_element(opt, &s, g, p, &m);
        t->param[e] = round_param(hp, pn, 0, E0 + (uint64_t)e);
        t->m32[e] = m;
    }
}

int q8o_onestate_sr_step(int opt, const q8o_tensor8* list, int n, const q8o_hparams* hp)
{
    uint64_t running = 0;
    for (int i = 0; i < n; ++i) {
        const q8o_tensor8* t = &list[i];
        uint64_t E0 = t->philox_offset >= 0 ? (uint64_t)t->philox_offset : running;
        if (t->m_codes) q8o_onestate8bit_tensor(opt, t, E0, hp);
        else q8o_onestate32_tensor(opt, t, E0, hp);
        running += (uint64_t)t->numel;
    }
    return 0;
}
