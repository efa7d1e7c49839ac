// ra_internal.h -- definitions shared by the host API and the kernels of libra.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/ra.h"

namespace ra {

// Tiling of the tensor-core path: 128 query rows per MMA tile (M), 128 keys per KV tile.
constexpr int kTile = 128;
// Workspace header: the device error word lives at offset 0; data starts here.
constexpr size_t kWsHeader = 256;
// Upper bound used by the automatic n_split choice (SM count of the target part).
constexpr int kAutoSplitSMs = 152;
// Default limit for every in-kernel wait.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// ---- token assignment (n = L / P tokens per shard) ----------------------------------
//   contiguous: local row a of shard i is token i*n + a
//   striped:    token a*P + i
//   zigzag:     2P chunks of c = n/2 tokens; rows [0, c) are chunk i, rows [c, 2c) are
//               chunk 2P-1-i (vanos001, section "The Causal-Mask Problem: Striped
//               Attention": two half-shards placed symmetrically near the two ends)
__host__ __device__ inline long long token_of(int layout, int i, long long a, long long n,
                                              int P) {
  if (layout == RA_LAYOUT_STRIPED) return a * P + i;
  if (layout == RA_LAYOUT_ZIGZAG) {
    const long long c = n >> 1;
    return a < c ? (long long)i * c + a : (2LL * P - 1 - i) * c + (a - c);
  }
  return (long long)i * n + a;
}

__host__ __device__ inline void shard_local_of(int layout, long long tok, long long n, int P,
                                               long long* shard, long long* local) {
  if (layout == RA_LAYOUT_STRIPED) {
    *shard = tok % P;
    *local = tok / P;
  } else if (layout == RA_LAYOUT_ZIGZAG) {
    const long long c = n >> 1, ch = tok / c;
    *shard = ch < P ? ch : 2LL * P - 1 - ch;
    *local = tok % c + (ch < P ? 0 : c);
  } else {
    *shard = tok / n;
    *local = tok % n;
  }
}

// For the blocked layouts (contiguous, zigzag): natural-order position of block t of
// shard i, counted in blocks of the same size (T blocks per shard, T even for zigzag).
// It increases with t, so the blocks of a shard that lie at or before a position g form
// a prefix, of length blocks_upto().
__host__ __device__ inline long long block_pos(int layout, int i, long long t, long long T,
                                               int P) {
  if (layout == RA_LAYOUT_ZIGZAG) {
    const long long Th = T >> 1;
    return t < Th ? (long long)i * Th + t : (2LL * P - 1 - i) * Th + (t - Th);
  }
  return (long long)i * T + t;
}

__host__ __device__ inline long long clamp_ll(long long x, long long lo, long long hi) {
  return x < lo ? lo : (x > hi ? hi : x);
}

// Number of blocks t of shard i with block_pos(i, t) <= g.
__host__ __device__ inline long long blocks_upto(int layout, int i, long long g, long long T,
                                                 int P) {
  if (layout == RA_LAYOUT_ZIGZAG) {
    const long long Th = T >> 1;
    return clamp_ll(g - (long long)i * Th + 1, 0, Th) +
           clamp_ll(g - (2LL * P - 1 - i) * Th + 1, 0, Th);
  }
  return clamp_ll(g - (long long)i * T + 1, 0, T);
}

// Number of tokens of shard j at or before token `tok` (any layout).
__host__ __device__ inline long long tokens_upto(int layout, int j, long long tok, long long n,
                                                 int P) {
  if (layout == RA_LAYOUT_STRIPED) return tok < j ? 0 : clamp_ll((tok - j) / P + 1, 0, n);
  return blocks_upto(layout, j, tok, n, P);   // blocks of one token
}

// A head's streamed operands at or above this size (half the L2) select the tile-outer
// walk for the striped layout: K and V in the forward, Q, dO and the fp32 dQ accumulator
// in the backward.
constexpr double kTileOuterBytes = 64.0 * 1024 * 1024;

// Ring schedule of one query-side unit of work: the query rows are the local 128-row
// tiles t0 .. t0+nq-1 of shard i; ring steps k0 .. k1-1 visit KV shard j = (i - k) mod P,
// and inside a step the KV tiles u = 0 .. u_end(j)-1 of that shard in order.
// Causal classification (per 128 x 128 tile, original token positions):
//   contiguous, zigzag: natural-order tile positions gq = block_pos(i, t),
//               gk = block_pos(j, u); skip gk > gq, diag gk == gq (mask b <= a);
//   striped:    skip u > t, diag u == t (mask inside: key b visible to query a iff
//               b < a, or b == a and j <= i), full u < t.
// In every layout the KV tiles of shard j that query tile t0+q sees form a prefix
// u < q_end(q, j), of which only the last can be the diagonal one (q_diag, -1 if none);
// u_end(j) is the longest such prefix over the unit's query tiles.
struct RingSched {
  int i, t0, nq, T, P, layout, causal, k0, k1;

  __host__ __device__ int j_of(int k) const {   // 0 <= i, k < P
    const int j = i - k;
    return j < 0 ? j + P : j;
  }
  __host__ __device__ int q_end(int q, int j) const {
    const int t = t0 + q;
    if (q >= nq || t >= T) return 0;
    if (!causal) return T;
    if (layout == RA_LAYOUT_STRIPED) return t + 1;
    return (int)blocks_upto(layout, j, block_pos(layout, i, t, T, P), T, P);
  }
  __host__ __device__ int q_diag(int q, int j) const {
    const int t = t0 + q;
    if (!causal || q >= nq || t >= T) return -1;
    if (layout == RA_LAYOUT_STRIPED) return t;
    const int e = q_end(q, j);
    return (e > 0 && block_pos(layout, j, e - 1, T, P) == block_pos(layout, i, t, T, P)) ? e - 1
                                                                                        : -1;
  }
  __host__ __device__ int u_end(int j) const {
    int e = 0;
    for (int q = 0; q < nq; ++q) {
      const int x = q_end(q, j);
      e = x > e ? x : e;
    }
    return e;
  }
  // longest u_end over the unit's ring steps
  __host__ __device__ int u_max() const {
    int e = 0;
    for (int k = k0; k < k1; ++k) {
      const int x = u_end(j_of(k));
      e = x > e ? x : e;
    }
    return e;
  }
};

// Backward schedule (KV-stationary ring): KV tile u of shard j meets the query shards
// i = (j + k) mod P in ring order.  For query tile t (128 rows) of shard i, key row b
// (0..127) is visible to query row a (0..127) iff a - b + delta >= 0 with
//   contiguous, zigzag: delta = 128 (block_pos(i, t) - block_pos(j, u))
//   striped:            delta = 128 (t - u) - (i < j)
// skip: delta < -127; full: delta >= 127 (or non-causal); otherwise masked.  Tile
// positions grow with t, so the visible query tiles of a shard are a suffix t >= t_lo.
struct BwdSched {
  int j, u, n, T, P, layout, causal;
  __host__ __device__ int i_of(int k) const {   // 0 <= j, k < P
    const int x = j + k;
    return x >= P ? x - P : x;
  }
  __host__ __device__ long long delta(int i, int t) const {
    if (layout == RA_LAYOUT_STRIPED) return 128LL * (t - u) - (i < j ? 1 : 0);
    return 128LL * (block_pos(layout, i, t, T, P) - block_pos(layout, j, u, T, P));
  }
  // first query tile with delta >= -127
  __host__ __device__ int t_lo(int i) const {
    if (!causal) return 0;
    if (layout != RA_LAYOUT_STRIPED)
      return (int)blocks_upto(layout, i, block_pos(layout, j, u, T, P) - 1, T, P);
    const long long num = 128LL * u + (i < j ? 1 : 0) - 127;
    if (num <= 0) return 0;
    const long long t = (num + 127) / 128;
    return t > T ? T : (int)t;
  }
};

struct FwdArgs {
  int B, H, D, P, layout, causal, block;
  int G;          // query heads per key/value head: query head h reads K/V head h / G
  int64_t L;
  int n;          // tokens per shard, L / P
  int T;          // 128-row tiles per shard
  int npair;      // CTAs per shard and head: ceil(T / 2)
  int n_split;    // ring-step groups
  float scale_log2;   // softmax scale * log2(e)
  void* out;          // fused mode output, bf16 or fp32
  int out_fp32;
  float* lse;
  float* o_part;      // split mode: [n_split][B, L, H, D] fp32
  float* lse_part;    // split mode: [n_split][B, H, L]
  unsigned long long* shard_work;   // [3][P] or null
  unsigned int* err;
  uint64_t wait_limit_ns;
};

struct BwdArgs {
  int B, H, D, P, layout, causal;
  int Hkv, G;     // key/value heads; query heads per key/value head (h = hk * G + g)
  int64_t L;
  int n, T;
  float scale;        // softmax scale
  float scale_log2;   // softmax scale * log2(e)
  const float* lse;   // -lse * log2(e), shard-major [B, H, P, n]
  const float* Dvec;  // -rowsum(dO * O), shard-major [B, H, P, n]
  float* dq_acc;      // [B, L, H, D] fp32
  void* dk;
  void* dv;
  unsigned int* err;
  uint64_t wait_limit_ns;
};

// Launchers (defined next to their kernels).
cudaError_t launch_fwd(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, cudaStream_t s);
cudaError_t launch_bwd(const BwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const CUtensorMap& tdo, cudaStream_t s);
cudaError_t launch_merge(int n_parts, const float* o_parts, const float* lse_parts, int B,
                         int64_t L, int H, int D, void* out, int out_fp32, float* lse,
                         cudaStream_t s);
cudaError_t launch_bwd_pre(const void* out, int out_fp32, const void* dout, const float* lse,
                           float* Dsm, float* L2sm, float* dq_acc, int B, int64_t L, int H, int D,
                           int P, int layout, cudaStream_t s);
cudaError_t launch_dq_convert(const float* dq_acc, void* dq, float scale, size_t n,
                              cudaStream_t s);
cudaError_t launch_selftest_timeout(unsigned int* err, uint64_t limit_ns, cudaStream_t s);
cudaError_t launch_selftest_exp2(const float* x, float* y_soft, float* y_hw, long long n,
                                 cudaStream_t s);

// Sets the text ra_last_error_message() returns on this thread.
void set_last_error_message(const char* msg);


}  // namespace ra
