// Predicates of the FA_DEBUG device checks (a build with -DFA_DEBUG=1).
//
// Each names a rule an access must follow on sm_103a; the checked build
// evaluates the rule before every access of that kind and, where it fails,
// records a bit in the device error word and skips the access instead of
// issuing it.  Plain C++ without CUDA types, so that the host tests compile
// and exercise the same functions with g++.
#pragma once
#include <stdint.h>

#ifdef __CUDACC__
#define FA_HD __host__ __device__
#else
#define FA_HD
#endif

namespace fa {

// Bits of the device error word set by the checked build (beside the wait
// time-out bits of common.cuh).
enum : unsigned int {
    kErrCheckTma = 1u << 16,   // tiled or bulk copy: coordinate, alignment, size
    kErrCheckTmem = 1u << 17,  // tcgen05.ld / st outside the warp's quadrant or the columns
    kErrCheckSmem = 1u << 18,  // hand-written shared-memory tile store, descriptor base
    kErrCheckTile = 1u << 19,  // work item decoded to a head or tile out of range
    kErrCheckMask = 0xFu << 16,
};

namespace chk {

// A tiled TMA copy (load, store or reduction) faults unless its innermost
// coordinate times the element size is a multiple of 16 bytes.  Every tile
// this library copies starts at a multiple of 16 elements, so the checked
// build demands that (elem_bytes = 1), which covers every element size.
FA_HD constexpr bool tma_inner_ok(long long x, int elem_bytes) {
    return ((x * elem_bytes) % 16) == 0;
}

// Tiled loads may start outside the tensor (the unit fills zeros there);
// stores and reductions start at non-negative coordinates.
FA_HD constexpr bool tma_store_ok(long long x, long long y, int elem_bytes) {
    return x >= 0 && y >= 0 && tma_inner_ok(x, elem_bytes);
}

// A 128-byte-swizzled tile (TMA destination or MMA operand) starts on a
// 1024-byte boundary of shared memory: the swizzle pattern repeats every
// 8 rows of 128 bytes and is anchored at the address bits above 1024.
FA_HD constexpr bool sw128_base_ok(uint32_t smem_addr) { return (smem_addr & 1023u) == 0; }

// Untiled bulk copies: both addresses 16-byte aligned, the size a positive
// multiple of 16 bytes.
FA_HD constexpr bool bulk_ok(uint64_t dst, uint64_t src, uint32_t bytes) {
    return (dst % 16) == 0 && (src % 16) == 0 && bytes > 0 && (bytes % 16) == 0;
}

// TMEM address = lane << 16 | column.  A warp's tcgen05.ld / st of the
// 32x32b shape reaches only the 32 lanes of its quadrant (warp index mod 4),
// and `ncols` 32-bit columns from `column` must lie inside the 512 columns
// of the SM's tensor memory.
constexpr uint32_t kTmemColumns = 512;
FA_HD constexpr bool tmem_ok(uint32_t taddr, uint32_t ncols, uint32_t warp_in_cta) {
    return (taddr >> 16) == 32u * (warp_in_cta % 4u) && (taddr & 0xFFFFu) + ncols <= kTmemColumns;
}

// [off, off + n) inside [0, size): a hand-written shared-memory store of a
// staging or operand tile, or a global row of an output.
FA_HD constexpr bool range_ok(long long off, long long n, long long size) {
    return off >= 0 && n >= 0 && off + n <= size;
}

// A work item's tile indices: head row in [0, heads), tile in [0, tiles).
FA_HD constexpr bool tile_ok(long long head, long long heads, long long tile, long long tiles) {
    return head >= 0 && head < heads && tile >= 0 && tile < tiles;
}

}  // namespace chk
}  // namespace fa
