// ra_aux.cu -- bandwidth-bound kernels around the tensor-core kernels:
//   * merge of normalised partials (O_g, lse_g) into (O, lse);
//   * backward preprocess D = rowsum(dO * O) (labhub, section "逆伝播での KV 再循環");
//   * fp32 dQ accumulator -> bf16 dQ with the softmax scale folded in;
//   * the bounded-wait self-test kernel.
// All of them stream rows of D contiguous elements with 16-byte vector accesses.
#include <cuda_bf16.h>

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

// One warp per output row (b, token, h); each lane owns 4 consecutive features per
// 128-feature chunk.  Weights exp(lse_g - max) are computed by every lane (n is small).
__global__ void __launch_bounds__(256)
    merge_kernel(int n_parts, const float* __restrict__ o_parts,
                 const float* __restrict__ lse_parts, int B, long long L, int H, int D,
                 void* out, int out_fp32, float* lse) {
  const long long rows = (long long)B * L * H;
  const long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  const int h = (int)(row % H);
  const long long bl = row / H;
  const long long tok = bl % L;
  const int b = (int)(bl / L);
  const size_t lidx = ((size_t)b * H + h) * L + tok;
  const size_t part_o = (size_t)rows * D;
  const size_t part_l = (size_t)B * H * L;
  float mx = kNegInf;
  for (int g = 0; g < n_parts; ++g) mx = fmaxf(mx, lse_parts[g * part_l + lidx]);
  float tot = 0.f;
  if (mx != kNegInf)
    for (int g = 0; g < n_parts; ++g) {
      const float l = lse_parts[g * part_l + lidx];
      if (l != kNegInf) tot += expf(l - mx);
    }
  const float inv = tot > 0.f ? 1.f / tot : 0.f;
  for (int d0 = lane * 4; d0 < D; d0 += 128) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (tot > 0.f)
      for (int g = 0; g < n_parts; ++g) {
        const float l = lse_parts[g * part_l + lidx];
        if (l == kNegInf) continue;
        const float w = expf(l - mx) * inv;
        const float4 o = __ldg(reinterpret_cast<const float4*>(o_parts + g * part_o +
                                                                (size_t)row * D + d0));
        acc.x += w * o.x;
        acc.y += w * o.y;
        acc.z += w * o.z;
        acc.w += w * o.w;
      }
    store4(out, out_fp32, (size_t)row * D + d0, acc);
  }
  if (lane == 0) lse[lidx] = tot > 0.f ? mx + logf(tot) : kNegInf;
}

// Backward preprocess, one warp per row (b, token, h):
//   nD[b, h, shard, local]    = -sum_d dO[b, token, h, d] * O[b, token, h, d]
//   nlse2[b, h, shard, local] = -lse[b, h, token] * log2(e)
// written shard-major so the values of one query tile are one contiguous block, and
// negated so that the backward's s*c - lse2 and dP - D are single packed FMAs/adds.
__global__ void __launch_bounds__(256)
    bwd_pre_kernel(const void* __restrict__ out, int out_fp32, const __nv_bfloat16* __restrict__ dout,
                   const float* __restrict__ lse, float* __restrict__ Dsm, float* __restrict__ L2sm,
                   int B, long long L, int H, int D, int P, int layout) {
  const long long rows = (long long)B * L * H;
  const long long row = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  float acc = 0.f;
  for (int d0 = lane * 4; d0 < D; d0 += 128) {
    const size_t e = (size_t)row * D + d0;
    const uint2 gw = __ldg(reinterpret_cast<const uint2*>(dout + e));
    const __nv_bfloat162 g01 = *reinterpret_cast<const __nv_bfloat162*>(&gw.x);
    const __nv_bfloat162 g23 = *reinterpret_cast<const __nv_bfloat162*>(&gw.y);
    float4 o;
    if (out_fp32) {
      o = __ldg(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(out) + e));
    } else {
      const uint2 ow = __ldg(reinterpret_cast<const uint2*>(
          reinterpret_cast<const __nv_bfloat16*>(out) + e));
      const float2 o01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ow.x));
      const float2 o23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ow.y));
      o = make_float4(o01.x, o01.y, o23.x, o23.y);
    }
    const float2 g0 = __bfloat1622float2(g01), g1 = __bfloat1622float2(g23);
    acc += g0.x * o.x + g0.y * o.y + g1.x * o.z + g1.y * o.w;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) {
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

unsigned grid_for(long long rows, int rows_per_block) {
  long long g = (rows + rows_per_block - 1) / rows_per_block;
  return (unsigned)(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t launch_merge(int n_parts, const float* o_parts, const float* lse_parts, int B,
                         int64_t L, int H, int D, void* out, int out_fp32, float* lse,
                         cudaStream_t s) {
  const long long rows = (long long)B * L * H;
  merge_kernel<<<grid_for(rows, 8), 256, 0, s>>>(n_parts, o_parts, lse_parts, B, L, H, D, out,
                                                 out_fp32, lse);
  return cudaGetLastError();
}

cudaError_t launch_bwd_pre(const void* out, int out_fp32, const void* dout, const float* lse,
                           float* Dsm, float* L2sm, int B, int64_t L, int H, int D, int P,
                           int layout, cudaStream_t s) {
  const long long rows = (long long)B * L * H;
  bwd_pre_kernel<<<grid_for(rows, 8), 256, 0, s>>>(
      out, out_fp32, reinterpret_cast<const __nv_bfloat16*>(dout), lse, Dsm, L2sm, B, L, H, D, P,
      layout);
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

cudaError_t launch_selftest_timeout(unsigned int* err, uint64_t limit_ns, cudaStream_t s) {
  selftest_timeout_kernel<<<1, 32, 0, s>>>(err, limit_ns);
  return cudaGetLastError();
}

}  // namespace ra
