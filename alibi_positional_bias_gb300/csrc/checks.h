// Predicates of the debug-checks build (compiled with -DALIBI_CHECKS).
//
// In that build the tensor-core kernels test every TMA coordinate, TMEM address
// and shared-memory operand against these predicates before the access. A failed
// test records ALIBI_DEV_CHECK in the device status word, with the check's id and
// the offending value in the site word ((id << 24) | (value & 0xFFFFFF)), and the
// access is skipped (a skipped load then shows up as a timeout of the wait that
// expected it). The normal build compiles none of this. Plain C++, so the host
// tests can pin the predicates without a GPU.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define ALIBI_HD __host__ __device__
#else
#define ALIBI_HD
#endif

namespace alibi {
namespace check {

enum : uint32_t {
    TMA_LOAD = 1,    // tiled load: x not on a 16-byte boundary, or destination misaligned / outside the window
    TMA_STORE = 2,   // tiled store: x misaligned or a negative coordinate, or source outside the window
    TMEM_COLS = 3,   // TMEM columns outside the CTA's allocation
    TMEM_LANES = 4,  // TMEM lanes outside the warp's quadrant
    SMEM_DESC = 5,   // MMA / copy operand outside the shared-memory window
};

// 16-bit elements: a tiled copy starts on a 16-byte boundary when x is a multiple of 8.
ALIBI_HD inline bool tma_x_aligned(int x) { return (x & 7) == 0; }

// A tiled store may not start at a negative coordinate (loads may: they fill).
ALIBI_HD inline bool tma_store_coords(int x, int y, int z) { return tma_x_aligned(x) && x >= 0 && y >= 0 && z >= 0; }

// `bytes` bytes at shared-memory address `saddr` lie inside [lo, hi) and start on an
// `align`-byte boundary (a power of two).
ALIBI_HD inline bool smem_range(uint32_t saddr, uint32_t bytes, uint32_t align, uint32_t lo, uint32_t hi)
{
    return (saddr & (align - 1)) == 0 && saddr >= lo && saddr <= hi && bytes <= hi - saddr;
}

// TMEM address = (lane << 16) | column. `width` columns from the address's column lie
// inside an allocation of `ncols` columns starting at column 0 (a CTA that takes the
// whole TMEM of its SM gets column 0).
ALIBI_HD inline bool tmem_cols(uint32_t taddr, uint32_t width, uint32_t ncols)
{
    const uint32_t col = taddr & 0xFFFFu;
    return col < ncols && width <= ncols - col;
}

// A warp may reach only the 32 TMEM lanes of its quadrant (warp index mod 4).
ALIBI_HD inline bool tmem_lanes(uint32_t taddr, uint32_t warp) { return (taddr >> 16) == 32u * (warp & 3u); }

// Columns an MMA writes: N of its kind::f16 instruction descriptor (N / 8 in bits 17-22).
ALIBI_HD inline uint32_t idesc_n(uint32_t idesc) { return ((idesc >> 17) & 0x3Fu) << 3; }

// Start address (bytes) in a shared-memory matrix descriptor (16-byte units, bits 0-13).
ALIBI_HD inline uint32_t desc_addr(uint64_t desc) { return static_cast<uint32_t>(desc & 0x3FFFu) << 4; }

// The site word a failed check records.
ALIBI_HD inline uint32_t site(uint32_t id, uint32_t value) { return (id << 24) | (value & 0xFFFFFFu); }

}  // namespace check
}  // namespace alibi
