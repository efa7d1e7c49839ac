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

enum TileClass : int { kSkip = 0, kFull = 1, kDiag = 2 };

// Ring schedule of one query-side unit of work: the query rows are the local 128-row
// tiles t0 .. t0+nq-1 of shard i; ring steps k0 .. k1-1 visit KV shard j = (i - k) mod P,
// and inside a step the KV tiles u = 0 .. u_end(j)-1 of that shard in order.
// Causal classification (per 128 x 128 tile, original token positions):
//   contiguous: global tiles gq = i*T + t, gk = j*T + u; skip gk > gq, diag gk == gq;
//   striped:    skip u > t, diag u == t (mask inside: key b visible to query a iff
//               b < a, or b == a and j <= i), full u < t.
struct RingSched {
  int i, t0, nq, T, P, layout, causal, k0, k1;

  __host__ __device__ int j_of(int k) const {
    int j = (i - k) % P;
    return j < 0 ? j + P : j;
  }
  __host__ __device__ int u_end(int j) const {
    if (!causal) return T;
    int tmax = t0 + nq - 1;
    if (tmax > T - 1) tmax = T - 1;
    if (layout == RA_LAYOUT_STRIPED) return tmax + 1;
    long long lim = (long long)(i - j) * T + tmax;
    if (lim < 0) return 0;
    return lim >= T ? T : (int)lim + 1;
  }
  __host__ __device__ int cls(int q, int j, int u) const {
    const int t = t0 + q;
    if (q >= nq || t >= T) return kSkip;
    if (!causal) return kFull;
    if (layout == RA_LAYOUT_STRIPED) return u < t ? kFull : (u == t ? kDiag : kSkip);
    const long long gq = (long long)i * T + t, gk = (long long)j * T + u;
    return gk < gq ? kFull : (gk == gq ? kDiag : kSkip);
  }
};

struct FwdArgs {
  int B, H, D, P, layout, causal, block;
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
                           float* Dsm, float* L2sm, int B, int64_t L, int H, int D, int P,
                           int layout, cudaStream_t s);
cudaError_t launch_dq_convert(const float* dq_acc, void* dq, float scale, size_t n,
                              cudaStream_t s);
cudaError_t launch_selftest_timeout(unsigned int* err, uint64_t limit_ns, cudaStream_t s);

// Sets the text ra_last_error_message() returns on this thread.
void set_last_error_message(const char* msg);

}  // namespace ra
