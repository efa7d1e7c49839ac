// ra_rows.cuh -- TMA load of 128 consecutive local rows of one shard, for every layout.
#pragma once

#include "ra_internal.h"
#include "ra_ptx.cuh"

namespace ra {

// The host views each bf16 [B, L, H, D] tensor as 5-D so that one box is 128 rows of one
// shard and 64 features of one head (make_rows_map):
//   striped    dims (D, H, P, n, B):   coordinates (d0, h, shard, local, b)
//   contiguous dims (D, H, n, P, B):   coordinates (d0, h, local, shard, b)
//   zigzag     dims (D, H, c, 2P, B):  coordinates (d0, h, local mod c, chunk, b), with
//              chunk = shard for local < c and 2P-1-shard otherwise; c = n/2 is a multiple
//              of 128, so a box never straddles the two chunks.
// W: the whole converged warp calls it and one elected lane issues the copy.
template <bool W = false>
__device__ __forceinline__ void load_rows(void* dst, const CUtensorMap* m, uint64_t* bar,
                                          int layout, int d0, int h, int shard, int local0,
                                          int b, int n, int P) {
  int c2 = shard, c3 = local0;                  // striped: (shard, local)
  if (layout == RA_LAYOUT_ZIGZAG) {
    const int c = n >> 1;
    const bool lo = local0 < c;
    c2 = lo ? local0 : local0 - c;
    c3 = lo ? shard : 2 * P - 1 - shard;
  } else if (layout != RA_LAYOUT_STRIPED) {     // contiguous: (local, shard)
    c2 = local0;
    c3 = shard;
  }
  if (W) tma_load_5d_w(dst, m, bar, d0, h, c2, c3, b);
  else tma_load_5d(dst, m, bar, d0, h, c2, c3, b);
}

// The box load_rows reads (64 features from d0, 128 local rows from local0, one head,
// shard and batch) lies inside a [B, P * n, heads, D] tensor's shard view.
__host__ __device__ inline bool rows_box_ok(int d0, int h, int shard, int local0, int b, int n,
                                            int P, int heads, int B, int D) {
  return d0 >= 0 && d0 + 64 <= D && h >= 0 && h < heads && shard >= 0 && shard < P &&
         local0 >= 0 && local0 + 128 <= n && b >= 0 && b < B;
}

}  // namespace ra
