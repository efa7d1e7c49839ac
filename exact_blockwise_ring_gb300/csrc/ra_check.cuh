// ra_check.cuh -- range checks of the checked build (compiled with -DRA_CHECKS).
//
// Tile and TMA box coordinates, TMEM columns and lane quarters, shared-memory operand
// offsets, global element indices and the per-role item counts are tested before use.
// A violation sets a bit of the workspace error word and the access is skipped, so the
// kernel leaves through its normal exit (no trap, no fault; a wait that can then no longer
// complete gives up after its time limit) and ra_check_error() reports RA_ERR_CHECK.  In
// the normal build kChecked is false and every check compiles to nothing.
#pragma once

#include <cstdint>

namespace ra {

constexpr uint32_t kChkTma = 0x100u;      // TMA box outside its tensor view, or a bad stage
constexpr uint32_t kChkTmem = 0x200u;     // TMEM column range or lane quarter outside bounds
constexpr uint32_t kChkSmem = 0x400u;     // shared-memory operand outside the kernel's layout
constexpr uint32_t kChkGlobal = 0x800u;   // global element index outside its tensor
constexpr uint32_t kChkSched = 0x1000u;   // the roles of a CTA disagree on its item count
constexpr uint32_t kChkMask = 0x1f00u;

#ifdef RA_CHECKS
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif

// True if `ok` (always true in the normal build); otherwise records `bit` in *err.
__device__ __forceinline__ bool check(unsigned int* err, bool ok, uint32_t bit) {
  if (kChecked && !ok) {
    atomicOr(err, bit);
    return false;
  }
  return true;
}

// A TMEM address (lane << 16 | column) of a 32-lane access by warp `warp` that touches
// columns [col, col + ncols): inside the 512-column allocation and in the warp's own lane
// quarter (warp mod 4), which is the only one tcgen05.ld/st can reach.
__device__ __forceinline__ bool tmem_ok(uint32_t taddr, uint32_t tbase, int ncols, int warp) {
  const uint32_t col = (taddr & 0xffffu) - (tbase & 0xffffu);
  const uint32_t lane = taddr >> 16;
  return col + (uint32_t)ncols <= 512u && lane == (uint32_t)(warp & 3) * 32u;
}

}  // namespace ra
