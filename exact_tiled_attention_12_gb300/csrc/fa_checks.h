// fa_checks.h — the bounds and alignment predicates of the debug build.
//
// A library built with FA_DEBUG_CHECKS (libfa_debug.so) evaluates these before
// every TMA tile load, bulk copy, tensor-memory load or store and MMA
// destination in its tensor-core kernels.  A failed check records a fault code
// in the library's fault word, raises the CTA's abort flag and skips the
// access (no trap, no device assert); the CTA's bounded waits then unwind it
// and fa_sync_status() reports FA_ERR_BOUNDS.  In the release build the checks
// compile to nothing.
//
// The predicates are plain functions of integers so that host code (and the
// host-side tests) can evaluate exactly what the kernels evaluate.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define FA_HD __host__ __device__ __forceinline__
#else
#define FA_HD inline
#endif

namespace fa {

#ifdef FA_DEBUG_CHECKS
constexpr bool kDebugChecks = true;
#else
constexpr bool kDebugChecks = false;
#endif

// Fault codes of failed checks: 0xC000 | kind << 8 | call site.
constexpr uint32_t kCheckBase = 0xC000u;
enum CheckKind : uint32_t {
  kChkTmaX = 1,      // innermost TMA coordinate not on a 16-byte boundary, or outside the row
  kChkTmaRows = 2,   // TMA box rows outside the tensor (2-D row view) or head index out of range (3-D)
  kChkSmem = 3,      // shared-memory destination or operand outside the dynamic allocation or misaligned
  kChkTmem = 4,      // tensor-memory column range outside the allocation
  kChkBulk = 5,      // bulk copy not 16-byte aligned or of a size that is not a multiple of 16
};
FA_HD constexpr uint32_t check_code(uint32_t kind, uint32_t site) { return kCheckBase | (kind << 8) | (site & 0xFFu); }
FA_HD constexpr bool is_check_code(uint32_t code) { return (code & 0xF000u) == kCheckBase; }

// A TMA tile load of a box `box_cols` elements wide starting at column x of
// rows `width` elements wide (16-bit elements): x must start on a 16-byte
// boundary (a multiple of 8 elements) and the box must start inside the row.
FA_HD constexpr bool tma_x_ok(int x, int box_cols, int width) {
  return x >= 0 && (x % 8) == 0 && x < width && box_cols > 0;
}

// 2-D row view [rows, width]: box rows [y, y + box_rows) inside [0, rows).
FA_HD constexpr bool tma_rows_ok(long long y, int box_rows, long long rows) {
  return y >= 0 && box_rows > 0 && y + box_rows <= rows;
}

// 3-D view [heads, n, width]: a box of rows starting at `pos` of head z.  Rows
// past n read as zero (the ragged last tile), so only the start must lie
// inside the head.
FA_HD constexpr bool tma_head_ok(int pos, int n, int z, int heads) {
  return pos >= 0 && pos < n && z >= 0 && z < heads;
}

// `bytes` of shared memory at offset `off` from the dynamic allocation's base
// (of `size` bytes), starting on an `align`-byte boundary.
FA_HD constexpr bool smem_ok(uint32_t off, uint32_t bytes, uint32_t size, uint32_t align) {
  return bytes > 0 && off < size && bytes <= size - off && (off % align) == 0;
}

// Columns [col, col + ncols) of a tensor-memory allocation of `alloc` columns.
FA_HD constexpr bool tmem_ok(uint32_t col, uint32_t ncols, uint32_t alloc) {
  return ncols > 0 && col < alloc && ncols <= alloc - col;
}

// A bulk (non-tensor) copy: both addresses 16-byte aligned, size a positive
// multiple of 16.
FA_HD constexpr bool bulk_ok(uint64_t gaddr, uint32_t saddr, uint32_t bytes) {
  return (gaddr % 16) == 0 && (saddr % 16) == 0 && bytes > 0 && (bytes % 16) == 0;
}

}  // namespace fa
