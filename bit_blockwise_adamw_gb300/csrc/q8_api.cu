// q8_api.cu -- the extern "C" entry points declared in include/q8adamw.h:
// argument checks, step scalars, launch planning over tensor lists.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <limits>
#include <memory>
#include <string>

#include "q8_internal.h"

namespace {

thread_local std::string g_error;

int fail(int code, const std::string& msg)
{
    g_error = msg;
    return code;
}

int cuda_fail(cudaError_t err, const char* where)
{
    return fail(Q8_ERR_CUDA, std::string(where) + ": " + cudaGetErrorString(err));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

constexpr int64_t kMaxNumel = int64_t(1) << 40;

std::string at(const char* what, int i)
{
    char buf[96];
    std::snprintf(buf, sizeof(buf), "%s (tensor %d)", what, i);
    return buf;
}

// Step scalars: formed in double from the hyper-parameters, rounded once to
// float.  beta^t is libm pow in double.  The fast mode (exact = 0) is taken
// only where its error bound holds: eps_t in [2^-36, 2^20] keeps the
// approximate reciprocal's argument normal and a subnormal v (flushed to zero)
// below half an ulp of eps_t; a_t <= 1 keeps the absolute error of a
// subnormal quotient, times a_t, below one fp32 step of the parameter
// (ratio2_approx).
int make_scalars(const q8_adamw_hparams* hp, q8::Scalars* s)
{
    if (!hp) return fail(Q8_ERR_NULL, "hparams is NULL");
    const double vals[5] = {hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay};
    for (double v : vals)
        if (!std::isfinite(v)) return fail(Q8_ERR_ARG, "hyper-parameters must be finite");
    if (hp->lr < 0.0) return fail(Q8_ERR_ARG, "lr must be >= 0");
    if (hp->beta1 < 0.0 || hp->beta1 >= 1.0) return fail(Q8_ERR_ARG, "beta1 must lie in [0, 1)");
    if (hp->beta2 < 0.0 || hp->beta2 >= 1.0) return fail(Q8_ERR_ARG, "beta2 must lie in [0, 1)");
    if (hp->eps < 0.0) return fail(Q8_ERR_ARG, "eps must be >= 0");
    if (hp->weight_decay < 0.0) return fail(Q8_ERR_ARG, "weight_decay must be >= 0");
    if (hp->step < 1 || hp->step > Q8_MAX_STEP) return fail(Q8_ERR_ARG, "step must lie in [1, 2^31)");
    if (hp->sr != 0 && hp->sr != 1) return fail(Q8_ERR_ARG, "sr must be 0 or 1");
    if (hp->exact != 0 && hp->exact != 1) return fail(Q8_ERR_ARG, "exact must be 0 or 1");
    const double t = static_cast<double>(hp->step);
    const double bc1 = 1.0 - std::pow(hp->beta1, t);
    const double bc2 = 1.0 - std::pow(hp->beta2, t);
    const double root_bc2 = std::sqrt(bc2);
    s->b1 = static_cast<float>(hp->beta1);
    s->omb1 = static_cast<float>(1.0 - hp->beta1);
    s->b2 = static_cast<float>(hp->beta2);
    s->omb2 = static_cast<float>(1.0 - hp->beta2);
    s->eps_t = static_cast<float>(hp->eps * root_bc2);
    s->step_size = static_cast<float>(hp->lr * root_bc2 / bc1);
    s->decay = static_cast<float>(1.0 - hp->lr * hp->weight_decay);
    s->key = q8::philox_key(hp->seed, static_cast<uint32_t>(hp->step));
    s->sr = hp->sr;
    s->fast_div = (s->eps_t >= 0x1p-100f && s->eps_t <= 0x1p20f) ? 1 : 0;
    s->approx = (hp->exact == 0 && s->eps_t >= 0x1p-36f && s->eps_t <= 0x1p20f && s->step_size <= 1.0f) ? 1 : 0;
    s->cancel = s->step_size * 0x1p-9f;
    s->two16 = 65536u;
    return Q8_OK;
}

int check_offset(int64_t e0, int64_t numel, int i)
{
    if (e0 > (int64_t(1) << 62) - numel) return fail(Q8_ERR_SIZE, at("philox_offset + numel exceeds 2^62", i));
    return Q8_OK;
}

int check_common(double lr, double wd, int64_t step, int32_t sr)
{
    if (!std::isfinite(lr) || !std::isfinite(wd)) return fail(Q8_ERR_ARG, "hyper-parameters must be finite");
    if (lr < 0.0) return fail(Q8_ERR_ARG, "lr must be >= 0");
    if (wd < 0.0) return fail(Q8_ERR_ARG, "weight_decay must be >= 0");
    if (step < 1 || step > Q8_MAX_STEP) return fail(Q8_ERR_ARG, "step must lie in [1, 2^31)");
    if (sr != 0 && sr != 1) return fail(Q8_ERR_ARG, "sr must be 0 or 1");
    return Q8_OK;
}

int check_beta(double b, const char* what)
{
    if (!std::isfinite(b) || b < 0.0 || b >= 1.0) return fail(Q8_ERR_ARG, std::string(what) + " must lie in [0, 1)");
    return Q8_OK;
}

// Momentum / Lion over a list: validate, then launch chunks of up to kMaxList
// entries (8-bit state on step1_kernel, fp32 state on step1_32_kernel).
int onestate_step(int opt, const q8_tensor8* list, int ntensors, const q8::Scalars1& s, cudaStream_t stream)
{
    if (ntensors < 0) return fail(Q8_ERR_SIZE, "ntensors must be >= 0");
    if (ntensors > 0 && !list) return fail(Q8_ERR_NULL, "list is NULL");
    int64_t running = 0;
    int rc;
    for (int i = 0; i < ntensors; ++i) {
        const q8_tensor8& t = list[i];
        if (t.numel < 0 || t.numel >= kMaxNumel) return fail(Q8_ERR_SIZE, at("numel must lie in [0, 2^40)", i));
        const int64_t e0 = t.philox_offset >= 0 ? t.philox_offset : running;
        running += t.numel;
        if (t.numel == 0) continue;
        if ((rc = check_offset(e0, t.numel, i)) != Q8_OK) return rc;
        if (!t.param || !t.grad) return fail(Q8_ERR_NULL, at("param and grad must be non-NULL", i));
        if (!aligned(t.param, 16) || !aligned(t.grad, 16))
            return fail(Q8_ERR_ALIGN, at("param and grad must be 16-byte aligned", i));
        if (t.v_codes || t.v_absmax || t.v32)
            return fail(Q8_ERR_ARG, at("one-state optimizers take no second-moment state", i));
        if (t.m_codes) {
            if (t.m32) return fail(Q8_ERR_ARG, at("an entry carries either 8-bit or fp32 state", i));
            if (!t.m_absmax) return fail(Q8_ERR_NULL, at("m_absmax must be non-NULL", i));
            if (!aligned(t.m_codes, 16) || !aligned(t.m_absmax, 4))
                return fail(Q8_ERR_ALIGN, at("codes must be 16-byte and absmax 4-byte aligned", i));
        } else {
            if (!t.m32) return fail(Q8_ERR_NULL, at("state pointers (m_codes or m32) are NULL", i));
            if (t.numel >= q8::kSmall) return fail(Q8_ERR_SIZE, at("fp32 state needs numel < 4096", i));
            if (!aligned(t.m32, 16)) return fail(Q8_ERR_ALIGN, at("m32 must be 16-byte aligned", i));
        }
    }
    if (ntensors == 0) return Q8_OK;
    const q8::DevTables* tab = nullptr;
    cudaError_t err = q8::device_tables(&tab);
    if (err != cudaSuccess) return cuda_fail(err, "device set-up");

    std::unique_ptr<q8::Step1Args> big(new q8::Step1Args());
    std::unique_ptr<q8::Step1_32Args> small(new q8::Step1_32Args());
    big->s = s;
    big->tab = tab;
    big->nt = 0;
    big->blk_start[0] = 0;
    small->s = s;
    small->nt = 0;
    auto flush_big = [&]() -> cudaError_t {
        if (big->nt == 0) return cudaSuccess;
        big->nblocks = big->blk_start[big->nt];
        const cudaError_t e = q8::launch_step1(opt, *big, stream);
        big->nt = 0;
        big->blk_start[0] = 0;
        return e;
    };
    auto flush_small = [&]() -> cudaError_t {
        if (small->nt == 0) return cudaSuccess;
        const cudaError_t e = q8::launch_step1_32(opt, *small, stream);
        small->nt = 0;
        return e;
    };
    running = 0;
    for (int i = 0; i < ntensors; ++i) {
        const q8_tensor8& t = list[i];
        const uint64_t e0 = static_cast<uint64_t>(t.philox_offset >= 0 ? t.philox_offset : running);
        running += t.numel;
        if (t.numel == 0) continue;
        if (t.m_codes) {
            const int64_t nb = (t.numel + q8::kBlock - 1) / q8::kBlock;
            if (big->nt == q8::kMaxList ||
                static_cast<int64_t>(big->blk_start[big->nt]) + nb > std::numeric_limits<int32_t>::max()) {
                if ((err = flush_big()) != cudaSuccess) return cuda_fail(err, "one-state step launch");
            }
            q8::Desc8& d = big->d[big->nt];
            d.p = t.param;
            d.g = t.grad;
            d.mq = t.m_codes;
            d.vq = nullptr;
            d.ma = t.m_absmax;
            d.va = nullptr;
            d.n = t.numel;
            d.e0 = e0;
            big->blk_start[big->nt + 1] = big->blk_start[big->nt] + static_cast<int32_t>(nb);
            ++big->nt;
        } else {
            if (small->nt == q8::kMaxList) {
                if ((err = flush_small()) != cudaSuccess) return cuda_fail(err, "one-state step launch");
            }
            q8::Desc32& d = small->d[small->nt++];
            d.p = t.param;
            d.g = t.grad;
            d.m = t.m32;
            d.v = nullptr;
            d.n = t.numel;
            d.e0 = e0;
        }
    }
    if ((err = flush_big()) != cudaSuccess) return cuda_fail(err, "one-state step launch");
    if ((err = flush_small()) != cudaSuccess) return cuda_fail(err, "one-state step launch");
    return Q8_OK;
}

void fill_common(q8::Scalars1& s, double lr, double wd, int64_t step, uint64_t seed, int32_t sr)
{
    s.lr_neg = static_cast<float>(-lr);
    s.decay = static_cast<float>(1.0 - lr * wd);
    s.wd = static_cast<float>(wd);
    s.key = q8::philox_key(seed, static_cast<uint32_t>(step));
    s.sr = sr;
}

}  // namespace

extern "C" {

int q8_abi_version(void) { return 5; }

const char* q8_last_error(void) { return g_error.c_str(); }

int q8_prepare_device(void)
{
    const q8::DevTables* tab = nullptr;
    cudaError_t err = q8::device_tables(&tab);
    if (err == cudaSuccess) err = q8::prepare_step8();
    if (err == cudaSuccess) err = q8::prepare_step1();
    if (err == cudaSuccess) err = q8::prepare_step16();
    if (err == cudaSuccess) err = q8::prepare_codec();
    if (err != cudaSuccess) return cuda_fail(err, "q8_prepare_device");
    return Q8_OK;
}

int q8_codebook_init(int kind, float* out)
{
    if (!out) return fail(Q8_ERR_NULL, "out is NULL");
    if (kind != Q8_SIGNED && kind != Q8_UNSIGNED) return fail(Q8_ERR_ARG, "kind must be Q8_SIGNED or Q8_UNSIGNED");
    q8::build_codebook(kind, out);
    return Q8_OK;
}

int q8_blockwise_quantize(const float* x, uint8_t* codes, float* absmax, int64_t n, int kind,
                          q8_stream_t stream)
{
    if (n < 0 || n >= kMaxNumel) return fail(Q8_ERR_SIZE, "n must lie in [0, 2^40)");
    if (kind != Q8_SIGNED && kind != Q8_UNSIGNED) return fail(Q8_ERR_ARG, "kind must be Q8_SIGNED or Q8_UNSIGNED");
    if (n == 0) return Q8_OK;
    if (!x || !codes || !absmax) return fail(Q8_ERR_NULL, "x, codes and absmax must be non-NULL");
    if (!aligned(x, 16) || !aligned(codes, 16) || !aligned(absmax, 4))
        return fail(Q8_ERR_ALIGN, "x and codes must be 16-byte aligned, absmax 4-byte aligned");
    const q8::DevTables* tab = nullptr;
    cudaError_t err = q8::device_tables(&tab);
    if (err != cudaSuccess) return cuda_fail(err, "device set-up");
    err = q8::launch_quantize(x, codes, absmax, n, kind, tab, stream);
    if (err != cudaSuccess) return cuda_fail(err, "q8_blockwise_quantize launch");
    return Q8_OK;
}

int q8_blockwise_dequantize(const uint8_t* codes, const float* absmax, float* x, int64_t n,
                            int kind, q8_stream_t stream)
{
    if (n < 0 || n >= kMaxNumel) return fail(Q8_ERR_SIZE, "n must lie in [0, 2^40)");
    if (kind != Q8_SIGNED && kind != Q8_UNSIGNED) return fail(Q8_ERR_ARG, "kind must be Q8_SIGNED or Q8_UNSIGNED");
    if (n == 0) return Q8_OK;
    if (!x || !codes || !absmax) return fail(Q8_ERR_NULL, "x, codes and absmax must be non-NULL");
    if (!aligned(x, 16) || !aligned(codes, 16) || !aligned(absmax, 4))
        return fail(Q8_ERR_ALIGN, "x and codes must be 16-byte aligned, absmax 4-byte aligned");
    const q8::DevTables* tab = nullptr;
    cudaError_t err = q8::device_tables(&tab);
    if (err != cudaSuccess) return cuda_fail(err, "device set-up");
    err = q8::launch_dequantize(codes, absmax, x, n, kind, tab, stream);
    if (err != cudaSuccess) return cuda_fail(err, "q8_blockwise_dequantize launch");
    return Q8_OK;
}

int q8_selftest_sqrt_div(uint64_t* counts, q8_stream_t stream)
{
    if (!counts) return fail(Q8_ERR_NULL, "counts is NULL");
    if (!aligned(counts, 8)) return fail(Q8_ERR_ALIGN, "counts must be 8-byte aligned");
    const cudaError_t err = q8::launch_selftest_sqrt_div(counts, stream);
    if (err != cudaSuccess) return cuda_fail(err, "q8_selftest_sqrt_div launch");
    return Q8_OK;
}

int q8_philox_fill(uint64_t seed, uint32_t step, uint32_t stream_id, uint64_t offset, int64_t n,
                   uint16_t* out, q8_stream_t stream)
{
    if (n < 0 || n >= kMaxNumel) return fail(Q8_ERR_SIZE, "n must lie in [0, 2^40)");
    if (offset > (uint64_t(1) << 62)) return fail(Q8_ERR_SIZE, "offset must be <= 2^62");
    if (n == 0) return Q8_OK;
    if (!out) return fail(Q8_ERR_NULL, "out is NULL");
    if (!aligned(out, 2)) return fail(Q8_ERR_ALIGN, "out must be 2-byte aligned");
    const cudaError_t err = q8::launch_philox_fill(q8::philox_key(seed, step), stream_id, offset, n, out, stream);
    if (err != cudaSuccess) return cuda_fail(err, "q8_philox_fill launch");
    return Q8_OK;
}

int adamw8bit_sr_step(const q8_tensor8* list, int ntensors, const q8_adamw_hparams* hp,
                      q8_stream_t stream)
{
    q8::Scalars s;
    int rc = make_scalars(hp, &s);
    if (rc != Q8_OK) return rc;
    if (ntensors < 0) return fail(Q8_ERR_SIZE, "ntensors must be >= 0");
    if (ntensors > 0 && !list) return fail(Q8_ERR_NULL, "list is NULL");

    // validate everything before launching anything
    int64_t running = 0;
    for (int i = 0; i < ntensors; ++i) {
        const q8_tensor8& t = list[i];
        if (t.numel < 0 || t.numel >= kMaxNumel) return fail(Q8_ERR_SIZE, at("numel must lie in [0, 2^40)", i));
        const int64_t e0 = t.philox_offset >= 0 ? t.philox_offset : running;
        running += t.numel;
        if (t.numel == 0) continue;
        if ((rc = check_offset(e0, t.numel, i)) != Q8_OK) return rc;
        if (!t.param || !t.grad) return fail(Q8_ERR_NULL, at("param and grad must be non-NULL", i));
        if (!aligned(t.param, 16) || !aligned(t.grad, 16))
            return fail(Q8_ERR_ALIGN, at("param and grad must be 16-byte aligned", i));
        if (t.m_codes) {
            if (t.m32 || t.v32) return fail(Q8_ERR_ARG, at("an entry carries either 8-bit or fp32 state", i));
            if (!t.v_codes || !t.m_absmax || !t.v_absmax)
                return fail(Q8_ERR_NULL, at("8-bit state pointers must be non-NULL", i));
            if (!aligned(t.m_codes, 16) || !aligned(t.v_codes, 16) || !aligned(t.m_absmax, 4) ||
                !aligned(t.v_absmax, 4))
                return fail(Q8_ERR_ALIGN, at("codes must be 16-byte and absmax 4-byte aligned", i));
        } else {
            if (!t.m32 || !t.v32) return fail(Q8_ERR_NULL, at("state pointers (codes or m32/v32) are NULL", i));
            if (t.numel >= q8::kSmall) return fail(Q8_ERR_SIZE, at("fp32 state needs numel < 4096", i));
            if (!aligned(t.m32, 16) || !aligned(t.v32, 16))
                return fail(Q8_ERR_ALIGN, at("m32 and v32 must be 16-byte aligned", i));
        }
    }
    if (ntensors == 0) return Q8_OK;

    const q8::DevTables* tab = nullptr;
    cudaError_t err = q8::device_tables(&tab);
    if (err != cudaSuccess) return cuda_fail(err, "device set-up");

    std::unique_ptr<q8::Step8Args> big(new q8::Step8Args());
    std::unique_ptr<q8::Step32Args> small(new q8::Step32Args());
    big->s = s;
    big->tab = tab;
    small->s = s;
    auto flush_big = [&]() -> cudaError_t {
        if (big->nt == 0) return cudaSuccess;
        big->nblocks = big->blk_start[big->nt];
        const cudaError_t e = q8::launch_step8(*big, stream);
        big->nt = 0;
        big->blk_start[0] = 0;
        return e;
    };
    auto flush_small = [&]() -> cudaError_t {
        if (small->nt == 0) return cudaSuccess;
        const cudaError_t e = q8::launch_step32(*small, stream);
        small->nt = 0;
        return e;
    };

    big->nt = 0;
    big->blk_start[0] = 0;
    small->nt = 0;
    running = 0;
    for (int i = 0; i < ntensors; ++i) {
        const q8_tensor8& t = list[i];
        const uint64_t e0 = static_cast<uint64_t>(t.philox_offset >= 0 ? t.philox_offset : running);
        running += t.numel;
        if (t.numel == 0) continue;
        if (t.m_codes) {
            const int64_t nb = (t.numel + q8::kBlock - 1) / q8::kBlock;
            if (big->nt == q8::kMaxList ||
                static_cast<int64_t>(big->blk_start[big->nt]) + nb > std::numeric_limits<int32_t>::max()) {
                if ((err = flush_big()) != cudaSuccess) return cuda_fail(err, "adamw8bit_sr_step launch");
            }
            q8::Desc8& d = big->d[big->nt];
            d.p = t.param;
            d.g = t.grad;
            d.mq = t.m_codes;
            d.vq = t.v_codes;
            d.ma = t.m_absmax;
            d.va = t.v_absmax;
            d.n = t.numel;
            d.e0 = e0;
            big->blk_start[big->nt + 1] = big->blk_start[big->nt] + static_cast<int32_t>(nb);
            ++big->nt;
        } else {
            if (small->nt == q8::kMaxList) {
                if ((err = flush_small()) != cudaSuccess) return cuda_fail(err, "adamw8bit_sr_step launch");
            }
            q8::Desc32& d = small->d[small->nt++];
            d.p = t.param;
            d.g = t.grad;
            d.m = t.m32;
            d.v = t.v32;
            d.n = t.numel;
            d.e0 = e0;
        }
    }
    if ((err = flush_big()) != cudaSuccess) return cuda_fail(err, "adamw8bit_sr_step launch");
    if ((err = flush_small()) != cudaSuccess) return cuda_fail(err, "adamw8bit_sr_step launch");
    return Q8_OK;
}

int adamw_bf16_sr_step(const q8_tensor16* list, int ntensors, const q8_adamw_hparams* hp,
                       q8_stream_t stream)
{
    q8::Scalars s;
    int rc = make_scalars(hp, &s);
    if (rc != Q8_OK) return rc;
    if (ntensors < 0) return fail(Q8_ERR_SIZE, "ntensors must be >= 0");
    if (ntensors > 0 && !list) return fail(Q8_ERR_NULL, "list is NULL");
    int64_t running = 0;
    for (int i = 0; i < ntensors; ++i) {
        const q8_tensor16& t = list[i];
        if (t.numel < 0 || t.numel >= kMaxNumel) return fail(Q8_ERR_SIZE, at("numel must lie in [0, 2^40)", i));
        const int64_t e0 = t.philox_offset >= 0 ? t.philox_offset : running;
        running += t.numel;
        if (t.numel == 0) continue;
        if ((rc = check_offset(e0, t.numel, i)) != Q8_OK) return rc;
        if (!t.param || !t.grad || !t.m || !t.v) return fail(Q8_ERR_NULL, at("param, grad, m and v must be non-NULL", i));
        if (!aligned(t.param, 16) || !aligned(t.grad, 16) || !aligned(t.m, 16) || !aligned(t.v, 16))
            return fail(Q8_ERR_ALIGN, at("param, grad, m and v must be 16-byte aligned", i));
    }
    if (ntensors == 0) return Q8_OK;

    std::unique_ptr<q8::Step16Args> args(new q8::Step16Args());
    args->s = s;
    args->nt = 0;
    args->blk_start[0] = 0;
    cudaError_t err;
    auto flush = [&]() -> cudaError_t {
        if (args->nt == 0) return cudaSuccess;
        args->nblocks = args->blk_start[args->nt];
        const cudaError_t e = q8::launch_step16(*args, stream);
        args->nt = 0;
        args->blk_start[0] = 0;
        return e;
    };
    running = 0;
    for (int i = 0; i < ntensors; ++i) {
        const q8_tensor16& t = list[i];
        const uint64_t e0 = static_cast<uint64_t>(t.philox_offset >= 0 ? t.philox_offset : running);
        running += t.numel;
        if (t.numel == 0) continue;
        const int64_t nb = (t.numel + q8::kBlock - 1) / q8::kBlock;
        if (args->nt == q8::kMaxList ||
            static_cast<int64_t>(args->blk_start[args->nt]) + nb > std::numeric_limits<int32_t>::max()) {
            if ((err = flush()) != cudaSuccess) return cuda_fail(err, "adamw_bf16_sr_step launch");
        }
        q8::Desc16& d = args->d[args->nt];
        d.p = t.param;
        d.g = t.grad;
        d.m = t.m;
        d.v = t.v;
        d.n = t.numel;
        d.e0 = e0;
        args->blk_start[args->nt + 1] = args->blk_start[args->nt] + static_cast<int32_t>(nb);
        ++args->nt;
    }
    if ((err = flush()) != cudaSuccess) return cuda_fail(err, "adamw_bf16_sr_step launch");
    return Q8_OK;
}

int momentum8bit_sr_step(const q8_tensor8* list, int ntensors, const q8_momentum_hparams* hp,
                         q8_stream_t stream)
{
    if (!hp) return fail(Q8_ERR_NULL, "hparams is NULL");
    int rc = check_common(hp->lr, hp->weight_decay, hp->step, hp->sr);
    if (rc != Q8_OK) return rc;
    if ((rc = check_beta(hp->momentum, "momentum")) != Q8_OK) return rc;
    q8::Scalars1 s{};
    fill_common(s, hp->lr, hp->weight_decay, hp->step, hp->seed, hp->sr);
    s.a = static_cast<float>(hp->momentum);
    s.oma = static_cast<float>(1.0 - hp->momentum);
    s.b = 0.0f;
    s.omb = 0.0f;
    return onestate_step(q8::kMomentum, list, ntensors, s, stream);
}

int lion8bit_sr_step(const q8_tensor8* list, int ntensors, const q8_lion_hparams* hp, q8_stream_t stream)
{
    if (!hp) return fail(Q8_ERR_NULL, "hparams is NULL");
    int rc = check_common(hp->lr, hp->weight_decay, hp->step, hp->sr);
    if (rc != Q8_OK) return rc;
    if ((rc = check_beta(hp->beta1, "beta1")) != Q8_OK) return rc;
    if ((rc = check_beta(hp->beta2, "beta2")) != Q8_OK) return rc;
    q8::Scalars1 s{};
    fill_common(s, hp->lr, hp->weight_decay, hp->step, hp->seed, hp->sr);
    s.a = static_cast<float>(hp->beta1);
    s.oma = static_cast<float>(1.0 - hp->beta1);
    s.b = static_cast<float>(hp->beta2);
    s.omb = static_cast<float>(1.0 - hp->beta2);
    return onestate_step(q8::kLion, list, ntensors, s, stream);
}

}  // extern "C"
