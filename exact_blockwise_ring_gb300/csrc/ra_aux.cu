// ra_aux.cu -- bandwidth-bound kernels around the tensor-core kernels:
//   * merge of normalised partials (O_g, lse_g) into (O, lse);
//   * backward preprocess D = rowsum(dO * O) (labhub, section "逆伝播での KV 再循環");
//   * fp32 dQ accumulator -> bf16 dQ with the softmax scale folded in;
//   * the bounded-wait self-test kernel and the 2^x self-test kernel.
// All of them stream rows of D contiguous elements with 16-byte vector accesses.
#include <cuda_bf16.h>

#include "ra_exp2.cuh"
#include "ra_internal.h"
#include "ra_ptx.cuh"

namespace ra {

namespace {

constexpr float kNegInf = -__builtin_huge_valf();

__device__ __forceinline__ void store4(void* out, int out_fp32, size_t elem, float4 v) {
  if (out_fp32) {
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + elem) = v;
  } else {
    uint2 w;
    w.x = pack_bf16x2(v.x, v.y);
    w.y = pack_bf16x2(v.z, v.w);
    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(out) + elem) = w;
  }
}

// Merge of n_parts normalised partials.  Rows are taken in the order of the lse arrays,
// (b, h) major and token fastest, so that the lse values of neighbouring rows are
// neighbouring words (coalesced loads and stores) while each row's D outputs stay one
// contiguous run.  A row is handled by `lpr` lanes (D/8 rounded up to a power of two),
// each owning 8 consecutive features; the grid is capped and strides over the rows.  The
// first kPrefetch parts' outputs and lse values are loaded before any is used, so their
// DRAM latency overlaps; further parts stream after.
constexpr int kPrefetch = 4;

__global__ void __launch_bounds__(256)
    merge_kernel(int n_parts, const float* __restrict__ o_parts,
                 const float* __restrict__ lse_parts, int B, long long L, int H, int D, int lpr,
                 void* out, int out_fp32, float* lse) {
  const long long rows = (long long)B * L * H;
  const int rpb = 256 / lpr;                      // rows per block and pass
  const int sub = threadIdx.x % lpr;
  const bool act = 8 * sub < D;
  const size_t part_o = (size_t)rows * D;
  const size_t part_l = (size_t)rows;             // B * H * L
  const long long step = (long long)gridDim.x * rpb;
  for (long long r = (long long)blockIdx.x * rpb + threadIdx.x / lpr; r < rows; r += step) {
    // r is the lse index (b * H + h) * L + token
    const long long tok = r % L;
    const long long bh = r / L;
    const long long h = bh % H, b = bh / H;
    const size_t e = (((size_t)b * L + tok) * H + h) * D + 8 * sub;
    float4 pa[kPrefetch], pb[kPrefetch];
    float lv[kPrefetch];
#pragma unroll
    for (int g = 0; g < kPrefetch; ++g) {
      if (act && g < n_parts) {
        const float4* src = reinterpret_cast<const float4*>(o_parts + g * part_o + e);
        pa[g] = __ldg(src);
        pb[g] = __ldg(src + 1);
      } else {
        pa[g] = pb[g] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      lv[g] = g < n_parts ? __ldg(lse_parts + g * part_l + r) : kNegInf;
    }
    // fmaxf skips NaN operands, so a NaN lse (a part whose rows met a NaN input) is
    // noted separately and makes the row's output and lse NaN
    float mx = kNegInf;
    bool nan = false;
#pragma unroll
    for (int g = 0; g < kPrefetch; ++g) {
      mx = fmaxf(mx, lv[g]);
      nan |= lv[g] != lv[g];
    }
    for (int g = kPrefetch; g < n_parts; ++g) {
      const float l = __ldg(lse_parts + g * part_l + r);
      mx = fmaxf(mx, l);
      nan |= l != l;
    }
    float tot = nan ? __int_as_float(0x7fc00000) : 0.f;
    if (!nan && mx != kNegInf) {
#pragma unroll
      for (int g = 0; g < kPrefetch; ++g)
        if (lv[g] != kNegInf) tot += expf(lv[g] - mx);
      for (int g = kPrefetch; g < n_parts; ++g) {
        const float l = __ldg(lse_parts + g * part_l + r);
        if (l != kNegInf) tot += expf(l - mx);
      }
    }
    const float inv = tot > 0.f ? 1.f / tot : 0.f;
    if (act) {
      float4 a0 = make_float4(tot, tot, tot, tot), a1 = a0;   // NaN rows stay NaN
      if (tot > 0.f) {
        a0 = a1 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int g = 0; g < kPrefetch; ++g) {
          if (lv[g] == kNegInf) continue;   // skipped (or absent), whatever its partial holds
          const float w = expf(lv[g] - mx) * inv;
          a0.x += w * pa[g].x; a0.y += w * pa[g].y; a0.z += w * pa[g].z; a0.w += w * pa[g].w;
          a1.x += w * pb[g].x; a1.y += w * pb[g].y; a1.z += w * pb[g].z; a1.w += w * pb[g].w;
        }
        for (int g = kPrefetch; g < n_parts; ++g) {
          const float l = __ldg(lse_parts + g * part_l + r);
          if (l == kNegInf) continue;
          const float w = expf(l - mx) * inv;
          const float4* src = reinterpret_cast<const float4*>(o_parts + g * part_o + e);
          const float4 x0 = __ldg(src), x1 = __ldg(src + 1);
          a0.x += w * x0.x; a0.y += w * x0.y; a0.z += w * x0.z; a0.w += w * x0.w;
          a1.x += w * x1.x; a1.y += w * x1.y; a1.z += w * x1.z; a1.w += w * x1.w;
        }
      }
      store4(out, out_fp32, e, a0);
      store4(out, out_fp32, e + 4, a1);
    }
    if (sub == 0) lse[r] = tot > 0.f ? mx + logf(tot) : (nan ? tot : kNegInf);
  }
}

// Backward preprocess.  Per row (b, token, h):
//   nD[b, h, shard, local]    = -sum_d dO[b, token, h, d] * O[b, token, h, d]
//   nlse2[b, h, shard, local] = -lse[b, h, token] * log2(e)
//   dq_acc[b, token, h, :]    = 0          (the backward main kernel adds into it)
// nD and nlse2 are written shard-major so the values of one query tile are one contiguous
// block, and negated so that the backward's s*c - lse2 and dP - D are single packed
// FMAs/adds.  A row is handled by D/8 consecutive lanes (8 features each: one 16-byte
// load of dO, one or two of O, two 16-byte stores of zeros), so a warp covers 256/D rows
// per pass; the dot product is reduced with shuffles inside each lane group.
__global__ void __launch_bounds__(256)
    bwd_pre_kernel(const void* __restrict__ out, int out_fp32, const __nv_bfloat16* __restrict__ dout,
                   const float* __restrict__ lse, float* __restrict__ Dsm, float* __restrict__ L2sm,
                   float* __restrict__ dq_acc, int B, long long L, int H, int D, int P,
                   int layout) {
  const int lpr = D >> 3;                             // lanes per row (8 or 16)
  const long long rows = (long long)B * L * H;
  const long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) / lpr;
  const int sub = threadIdx.x % lpr;
  const bool live = row < rows;
  float acc = 0.f;
  if (live) {
    const size_t e = (size_t)row * D + 8 * sub;
    const uint4 gw = __ldg(reinterpret_cast<const uint4*>(dout + e));
    float o[8];
    if (out_fp32) {
      const float4 a = __ldg(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(out) + e));
      const float4 c = __ldg(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(out) + e) + 1);
      o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
      o[4] = c.x; o[5] = c.y; o[6] = c.z; o[7] = c.w;
    } else {
      const uint4 ow = __ldg(reinterpret_cast<const uint4*>(
          reinterpret_cast<const __nv_bfloat16*>(out) + e));
      const uint32_t ov[4] = {ow.x, ow.y, ow.z, ow.w};
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ov[x]));
        o[2 * x] = f.x;
        o[2 * x + 1] = f.y;
      }
    }
    const uint32_t gv[4] = {gw.x, gw.y, gw.z, gw.w};
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const float2 g = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gv[x]));
      acc += g.x * o[2 * x] + g.y * o[2 * x + 1];
    }
    float4* z = reinterpret_cast<float4*>(dq_acc + e);
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // lane groups are aligned to lpr (a power of two dividing 32): xor stays inside a group
  for (int off = lpr >> 1; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (live && sub == 0) {
    const int h = (int)(row % H);
    const long long bl = row / H;
    const long long tok = bl % L;
    const int b = (int)(bl / L);
    const long long n = L / P;
    long long shard, local;
    shard_local_of(layout, tok, n, P, &shard, &local);
    const size_t bh = (size_t)b * H + h;
    const size_t dst = (bh * P + shard) * n + local;
    Dsm[dst] = -acc;
    L2sm[dst] = -lse[bh * L + tok] * 1.4426950408889634f;
  }
}

// dq[e] = bf16(scale * dq_acc[e]), 8 elements per thread.
__global__ void __launch_bounds__(256)
    dq_convert_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ dq, float scale,
                      size_t n8) {
  for (size_t v = (size_t)blockIdx.x * blockDim.x + threadIdx.x; v < n8;
       v += (size_t)gridDim.x * blockDim.x) {
    const float4 a0 = __ldg(reinterpret_cast<const float4*>(acc) + 2 * v);
    const float4 a1 = __ldg(reinterpret_cast<const float4*>(acc) + 2 * v + 1);
    uint4 w;
    w.x = pack_bf16x2(a0.x * scale, a0.y * scale);
    w.y = pack_bf16x2(a0.z * scale, a0.w * scale);
    w.z = pack_bf16x2(a1.x * scale, a1.y * scale);
    w.w = pack_bf16x2(a1.z * scale, a1.w * scale);
    reinterpret_cast<uint4*>(dq)[v] = w;
  }
}

// One CTA waits on an mbarrier that nothing arrives on; the bounded wait gives up after
// `limit_ns`, records the timeout in the error word and the kernel returns normally.
__global__ void selftest_timeout_kernel(unsigned int* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const WaitCtx wc{&abort_flag, err, limit_ns};
    (void)mbar_wait(&bar, 0, wc);
  }
  __syncthreads();
}

// Both 2^x forms of the softmax kernels on the same inputs (a pair per thread).
__global__ void selftest_exp2_kernel(const float* __restrict__ x, float* __restrict__ y_soft,
                                     float* __restrict__ y_hw, long long n) {
  const long long i = 2 * ((long long)blockIdx.x * blockDim.x + threadIdx.x);
  if (i >= n) return;
  const float x0 = x[i], x1 = i + 1 < n ? x[i + 1] : 0.f;
  float s0, s1;
  f2_unpack(exp2_soft_x2(x0, x1), s0, s1);
  y_soft[i] = s0;
  y_hw[i] = ex2_approx(x0);
  if (i + 1 < n) {
    y_soft[i + 1] = s1;
    y_hw[i + 1] = ex2_approx(x1);
  }
}

unsigned grid_for(long long rows, int rows_per_block) {
  long long g = (rows + rows_per_block - 1) / rows_per_block;
  return (unsigned)(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t launch_merge(int n_parts, const float* o_parts, const float* lse_parts, int B,
                         int64_t L, int H, int D, void* out, int out_fp32, float* lse,
                         cudaStream_t s) {
  if (D % 8 != 0 || D < 8 || D > 256) return cudaErrorInvalidValue;
  const long long rows = (long long)B * L * H;
  int lpr = 1;
  while (lpr < D / 8) lpr <<= 1;
  // as many blocks as are resident at once on the current device (every SM full),
  // striding over the rows; looked up on every call (a few microseconds of host work)
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, merge_kernel, 256, 0);
  if (e != cudaSuccess) return e;
  const long long cap = (long long)sms * (per_sm > 0 ? per_sm : 1);
  unsigned grid = grid_for(rows, 256 / lpr);
  if ((long long)grid > cap) grid = (unsigned)cap;
  merge_kernel<<<grid, 256, 0, s>>>(n_parts, o_parts, lse_parts, B, L, H, D, lpr, out, out_fp32,
                                    lse);
  return cudaGetLastError();
}

cudaError_t launch_bwd_pre(const void* out, int out_fp32, const void* dout, const float* lse,
                           float* Dsm, float* L2sm, float* dq_acc, int B, int64_t L, int H, int D,
                           int P, int layout, cudaStream_t s) {
  if (D % 8 != 0 || D < 8 || D > 256 || (D & (D - 1)) != 0) return cudaErrorInvalidValue;
  const long long rows = (long long)B * L * H;
  bwd_pre_kernel<<<grid_for(rows, 256 / (D / 8)), 256, 0, s>>>(
      out, out_fp32, reinterpret_cast<const __nv_bfloat16*>(dout), lse, Dsm, L2sm, dq_acc, B, L,
      H, D, P, layout);
  return cudaGetLastError();
}

cudaError_t launch_dq_convert(const float* dq_acc, void* dq, float scale, size_t n,
                              cudaStream_t s) {
  const size_t n8 = n / 8;
  long long blocks = (long long)((n8 + 255) / 256);
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  dq_convert_kernel<<<(unsigned)blocks, 256, 0, s>>>(
      dq_acc, reinterpret_cast<__nv_bfloat16*>(dq), scale, n8);
  return cudaGetLastError();
}

cudaError_t launch_selftest_exp2(const float* x, float* y_soft, float* y_hw, long long n,
                                 cudaStream_t s) {
  selftest_exp2_kernel<<<grid_for((n + 1) / 2, 256), 256, 0, s>>>(x, y_soft, y_hw, n);
  return cudaGetLastError();
}

cudaError_t launch_selftest_timeout(unsigned int* err, uint64_t limit_ns, cudaStream_t s) {
  selftest_timeout_kernel<<<1, 32, 0, s>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace ra
