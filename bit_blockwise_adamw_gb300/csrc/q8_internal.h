// q8_internal.h -- declarations shared by the library's translation units:
// table layout, kernel argument blocks and host-side launchers.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "q8adamw.h"

namespace q8 {

// Blocking ("8-bit Optimizers via Block-wise Quantization", method bullets:
// 2048-element blocks).  The codec, BF16-state and fp32-state kernels use
// 256-thread CTAs with eight contiguous elements per thread (one 16-byte load
// of bf16 data, one Philox call); the 8-bit step kernels use their own
// 128-thread layout.
constexpr int kBlock = 2048;
constexpr int kThreads = 256;
constexpr int kVec = 8;
static_assert(kThreads * kVec == kBlock, "one block per CTA iteration");
constexpr int kWarps = kThreads / 32;
constexpr int kSmall = 4096;

// Search cells.  A magnitude |y| <= 1 falls in a cell given by its binade and
// the top seven mantissa bits (every 2^16 consecutive bit patterns share a
// cell); magnitudes below 2^-L form cell 0.  L is chosen so that no midpoint
// lies in cell 0 and the seven mantissa bits keep at most one midpoint in any
// cell, so the count of midpoints below |y| is
//   base(cell) + (|y| beyond the cell's midpoint).
// Entry layout (uint32): bits 0..7 = base count, bits 16..31 = the low 16 bits
// of the in-cell midpoint; a cell that holds none stores 0xFFFFFF00 | base.  The signed table
// counts only the positive midpoints (the book is odd-symmetric, so the sign
// is applied after the lookup); the unsigned table counts all of them.
// cell = max((|y| bits >> 16) + bias, 0).
constexpr int kCellShift = 16;
constexpr int kSignedL = 21;      // smallest signed midpoint is 5e-7 > 2^-21
constexpr int kUnsignedL = 25;    // smallest unsigned midpoint is 5e-8 > 2^-25
constexpr int kCellsSigned = 2 + kSignedL * 128;
constexpr int kCellsUnsigned = 2 + kUnsignedL * 128;
constexpr int kSignedCellBias = 1 - ((127 - kSignedL) << 7);
constexpr int kUnsignedCellBias = 1 - ((127 - kUnsignedL) << 7);
constexpr int kCellSEntries = kCellsSigned + 2;      // padded to a multiple of 4 entries

struct alignas(16) DevTables {
    float cs[256];                         // signed codebook (dequantize m)
    float cu[256];                         // unsigned codebook (dequantize v)
    uint32_t cell_s[kCellSEntries];        // positive midpoints 127..253, by |y|
    uint32_t cell_u[kCellsUnsigned];       // non-negative x only
};
static_assert(sizeof(DevTables) % 16 == 0, "tables are copied to shared memory 16 bytes at a time");

// Philox4x32-10 key schedule of one call (Salmon, Moraes, Dror, Shaw, SC'11):
// round r uses the key (k0 + r*0x9E3779B9, k1 + r*0xBB67AE85) mod 2^32, with
// (k0, k1) = (low, high) 32 bits of the seed.  Formed once on the host, so
// each round reads its key as a kernel-parameter operand.  `step` is counter
// word 2.
struct PhiloxKey {
    uint32_t kx[10], ky[10];
    uint32_t step;
};
PhiloxKey philox_key(uint64_t seed, uint32_t step);

// Step scalars formed on the host in double and rounded once to float.
struct Scalars {
    float b1, omb1, b2, omb2, eps_t, step_size, decay;
    PhiloxKey key;
    int32_t sr;
    int32_t fast_div;          // eps_t in [2^-100, 2^20]: the packed division may be used
    int32_t approx;            // the caller did not ask for exact, eps_t in [2^-36, 2^20] and
                               // step_size <= 1: the full blocks' parameter update may use
                               // the approximate square root and reciprocal (ratio2_approx)
    float cancel;              // step_size * 2^-9: the cancellation bound of the fast mode
    uint32_t two16;            // 65536, from the host: the AdamW kernel's low-half bf16
                               // unpack is a multiply by it, which runs on the FMA pipe
                               // (a shift would load the busier ALU pipe)
};

// Tensor lists travel as kernel parameters (no device allocation, no copy):
// at most kMaxList tensors per launch; longer lists take several launches.
constexpr int kMaxList = 448;

struct Desc8 {                 // one 8-bit-state tensor, 64 bytes
    uint16_t* p;
    const uint16_t* g;
    uint8_t* mq;
    uint8_t* vq;
    float* ma;
    float* va;
    int64_t n;
    uint64_t e0;               // Philox index of element 0
};

struct Step8Args {
    Scalars s;
    const DevTables* tab;
    int32_t nt;
    int32_t nblocks;                      // total 2048-blocks in this launch
    int32_t blk_start[kMaxList + 1];      // first global block of each tensor
    Desc8 d[kMaxList];
};

struct Desc32 {                // one fp32-state tensor (numel < 4096)
    uint16_t* p;
    const uint16_t* g;
    float* m;
    float* v;
    int64_t n;
    uint64_t e0;
};

struct Step32Args {
    Scalars s;
    int32_t nt;
    Desc32 d[kMaxList];
};

struct Desc16 {                // one bf16-state tensor
    uint16_t* p;
    const uint16_t* g;
    uint16_t* m;
    uint16_t* v;
    int64_t n;
    uint64_t e0;
};

struct Step16Args {
    Scalars s;
    int32_t nt;
    int32_t nblocks;
    int32_t blk_start[kMaxList + 1];
    Desc16 d[kMaxList];
};

// One-state optimizers (8-bit Momentum, 8-bit Lion): scalars rounded once to
// float on the host; the tensor list reuses Desc8 / Desc32 with only the
// first-moment fields set.
enum { kMomentum = 0, kLion = 1 };

struct Scalars1 {
    float lr_neg, a, oma, b, omb, decay, wd;
    PhiloxKey key;
    int32_t sr;
};

struct Step1Args {
    Scalars1 s;
    const DevTables* tab;
    int32_t nt;
    int32_t nblocks;
    int32_t blk_start[kMaxList + 1];
    Desc8 d[kMaxList];
};

struct Step1_32Args {
    Scalars1 s;
    int32_t nt;
    Desc32 d[kMaxList];
};

static_assert(sizeof(Step8Args) <= 32764, "kernel parameter space");
static_assert(sizeof(Step1Args) <= 32764, "kernel parameter space");
static_assert(sizeof(Step16Args) <= 32764, "kernel parameter space");
static_assert(sizeof(Step32Args) <= 32764, "kernel parameter space");

// Host-side table construction (q8_tables.cu).
void build_codebook(int kind, float out[256]);
// Device copy of the tables for the current device, set up on first use.
cudaError_t device_tables(const DevTables** out);

// Grid of a persistent kernel on the current device: SMs x resident CTAs of
// `kernel` at `threads` threads and `smem` bytes of dynamic shared memory.
// Worked out once per (kernel, device) under a lock (which also raises the
// kernel's dynamic shared-memory limit to `smem` on that device) and cached,
// so concurrent first calls from several host threads, and processes that
// drive several devices, each get their own device's figure.
cudaError_t persistent_grid(const void* kernel, int threads, size_t smem, int* grid);

// Work out (and cache) the launch configuration of every kernel of one
// translation unit on the current device, so that later launches do no set-up.
cudaError_t prepare_step8();
cudaError_t prepare_step1();
cudaError_t prepare_step16();
cudaError_t prepare_codec();

// Launchers (one per kernel; each returns cudaGetLastError()).
cudaError_t launch_step8(const Step8Args& a, cudaStream_t st);
cudaError_t launch_step32(const Step32Args& a, cudaStream_t st);
cudaError_t launch_step16(const Step16Args& a, cudaStream_t st);
cudaError_t launch_step1(int opt, const Step1Args& a, cudaStream_t st);
cudaError_t launch_step1_32(int opt, const Step1_32Args& a, cudaStream_t st);
cudaError_t launch_quantize(const float* x, uint8_t* codes, float* absmax, int64_t n, int kind,
                            const DevTables* tab, cudaStream_t st);
cudaError_t launch_dequantize(const uint8_t* codes, const float* absmax, float* x, int64_t n,
                              int kind, const DevTables* tab, cudaStream_t st);
cudaError_t launch_selftest_sqrt_div(uint64_t* counts, cudaStream_t st);
cudaError_t launch_philox_fill(const PhiloxKey& key, uint32_t stream_id, uint64_t offset, int64_t n,
                               uint16_t* out, cudaStream_t st);

}  // namespace q8
