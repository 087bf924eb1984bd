// q8_tables.cu -- codebooks, decision midpoints and the cell search table:
// built once on the host, uploaded once per device.
//
// Codebooks ("8-bit Optimizers via Block-wise Quantization", innovations list:
// dynamic tree quantization, extended to unipolar data).  Reading: after the
// sign, a run of e zero bits selects the decade 10^-e, an indicator bit
// follows, and the remaining f bits place the value linearly inside the
// decade at 10^-e * (0.1 + 0.9*(j+1)/2^f), j = 0..2^f-1.  Signed book: 7 bits
// after the sign (e = 0..6, f = 6-e), mirrored around zero, with a duplicate
// 1.0 at index 255 that the search never returns; unsigned book: 8 bits
// (e = 0..7, f = 7-e) and zero.  Listing the decades from the smallest
// (largest e) up gives the tables in ascending order directly.
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "q8_internal.h"

namespace q8 {

namespace {

// One decade's values, ascending, appended at out[pos...]; returns new pos.
int append_decade(int e, int f, float* out, int pos)
{
    int64_t scale = 10;
    for (int i = 0; i < e; ++i) scale *= 10;            // 10^(e+1)
    const int64_t den = scale << f;                      // 10^(e+1) * 2^f
    for (int j = 0; j < (1 << f); ++j) {
        const int64_t num = (int64_t(1) << f) + 9 * int64_t(j + 1);
        out[pos++] = static_cast<float>(static_cast<double>(num) / static_cast<double>(den));
    }
    return pos;
}

void build_midpoints(const float c[256], float mid[255])
{
    for (int j = 0; j < 255; ++j)
        mid[j] = static_cast<float>(0.5 * (static_cast<double>(c[j]) + static_cast<double>(c[j + 1])));
}

float bits_to_float(uint32_t u) { float f; std::memcpy(&f, &u, 4); return f; }
uint32_t float_to_bits(float f) { uint32_t u; std::memcpy(&u, &f, 4); return u; }

// Fill a cell table over magnitudes from the ascending midpoints mid[0..nmid)
// (all positive); returns false if a cell would hold more than one midpoint
// (the table could not then decide with one compare).
bool build_cells(const float* mid, int nmid, int L, int ncells, uint32_t* out)
{
    const uint32_t low = static_cast<uint32_t>(127 - L) << 23;
    for (int c = 0; c < ncells; ++c) {
        uint32_t a_lo, a_hi;                              // magnitude bit range
        if (c == 0) { a_lo = 0; a_hi = low - 1; }
        else {
            a_lo = low + (static_cast<uint32_t>(c - 1) << kCellShift);
            a_hi = a_lo + ((1u << kCellShift) - 1);
        }
        if (a_hi > 0x3F800000u) a_hi = 0x3F800000u;
        if (a_lo > a_hi) a_lo = a_hi;
        const float x_first = bits_to_float(a_lo);
        const float x_last = bits_to_float(a_hi);
        uint32_t base = 0;
        while (static_cast<int>(base) < nmid && mid[base] < x_first) ++base;
        int inside = 0;
        uint32_t ml = 0xFFFFu;
        for (int j = static_cast<int>(base); j < nmid && mid[j] <= x_last; ++j) {
            ++inside;
            ml = float_to_bits(mid[j]) & 0xFFFFu;
        }
        if (inside > 1 || (c == 0 && inside > 0)) return false;
        // a cell without a midpoint also sets bits 8..15, so that no key (at
        // most 0xFFFFFF00) ever compares above it
        out[c] = (ml << 16) | base | (inside ? 0u : 0xFF00u);
    }
    return true;
}

struct HostTables {
    DevTables t;
    bool ok = false;
    HostTables()
    {
        float mid_s[255], mid_u[255];
        build_codebook(Q8_SIGNED, t.cs);
        build_codebook(Q8_UNSIGNED, t.cu);
        build_midpoints(t.cs, mid_s);
        build_midpoints(t.cu, mid_u);
        std::memset(t.cell_s, 0, sizeof(t.cell_s));
        // signed book: positive midpoints mid[127..253] (mid[254] is the pad's
        // 1.0, never below any |y| <= 1); the book must be odd-symmetric
        bool symmetric = true;
        for (int i = 0; i < 127; ++i) symmetric = symmetric && mid_s[126 - i] == -mid_s[127 + i];
        ok = symmetric
          && build_cells(mid_s + 127, 127, kSignedL, kCellsSigned, t.cell_s)
          && build_cells(mid_u, 255, kUnsignedL, kCellsUnsigned, t.cell_u);
    }
};

const HostTables& host_tables()
{
    static const HostTables h;
    return h;
}

__device__ DevTables g_tables;

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
const DevTables* g_dev_ptr[kMaxDevices] = {};

// persistent_grid's cache: (kernel, device, threads, smem) -> grid.
std::mutex g_grid_mutex;
std::map<std::tuple<const void*, int, int, size_t>, int> g_grids;

}  // namespace

cudaError_t persistent_grid(const void* kernel, int threads, size_t smem, int* grid)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const auto key = std::make_tuple(kernel, dev, threads, smem);
    std::lock_guard<std::mutex> lock(g_grid_mutex);
    const auto it = g_grids.find(key);
    if (it != g_grids.end()) {
        *grid = it->second;
        return cudaSuccess;
    }
    if (smem > 0) {
        err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (err != cudaSuccess) return err;
    }
    int sms = 0, per_sm = 0;
    if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
    if ((err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem)) != cudaSuccess)
        return err;
    if (sms <= 0 || per_sm <= 0) return cudaErrorInvalidConfiguration;
    g_grids.emplace(key, sms * per_sm);
    *grid = sms * per_sm;
    return cudaSuccess;
}

void build_codebook(int kind, float out[256])
{
    if (kind == Q8_UNSIGNED) {
        int pos = 0;
        out[pos++] = 0.0f;
        for (int e = 7; e >= 0; --e) pos = append_decade(e, 7 - e, out, pos);
    } else {
        float mag[127];
        int pos = 0;
        for (int e = 6; e >= 0; --e) pos = append_decade(e, 6 - e, mag, pos);
        for (int i = 0; i < 127; ++i) {
            out[128 + i] = mag[i];
            out[126 - i] = -mag[i];
        }
        out[127] = 0.0f;
        out[255] = 1.0f;
    }
}

cudaError_t device_tables(const DevTables** out)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_dev_ptr[dev]) {
        const HostTables& h = host_tables();
        if (!h.ok) return cudaErrorInvalidValue;
        err = cudaMemcpyToSymbol(g_tables, &h.t, sizeof(DevTables));
        if (err != cudaSuccess) return err;
        err = cudaDeviceSynchronize();
        if (err != cudaSuccess) return err;
        void* p = nullptr;
        err = cudaGetSymbolAddress(&p, g_tables);
        if (err != cudaSuccess) return err;
        g_dev_ptr[dev] = static_cast<const DevTables*>(p);
    }
    *out = g_dev_ptr[dev];
    return cudaSuccess;
}

}  // namespace q8
