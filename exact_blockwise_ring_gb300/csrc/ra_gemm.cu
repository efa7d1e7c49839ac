// ra_gemm.cu -- the dense kernels of the blockwise transformer layer (labhub "Ring Attention
// 論文分析", section "BPT の Feedforward 融合"): a tcgen05 GEMM for its Linear layers with
// the elementwise work fused into the epilogue, and a row LayerNorm.
//
// GEMM: out[M, N] = epilogue(A[M, K] B[N, K]^T + bias[N]), A and B bf16 row-major (B is a
// torch.nn.Linear weight [out_features, in_features]), fp32 accumulation in TMEM.
//   kEpiBias          out bf16 = acc + bias
//   kEpiBiasGelu      out bf16 = GELU(acc + bias), GELU(z) = z/2 (1 + erf(z / sqrt 2))
//   kEpiBiasResidual  out fp32 = acc + bias + residual[M, N] (bf16)
// Persistent: one CTA per SM walks output tiles of 128 x 256.  Roles (192 threads):
//   warp 0      TMA producer: per 64-wide K step one A box (128 x 64) and one B box
//               (256 x 64), 128-byte swizzled, into a kStages-deep ring shared by all of
//               the CTA's tiles
//   warp 1      TMEM owner (512 columns: two 256-column accumulators) and tcgen05.mma
//               issuer: M = 128, N = 256, K = 16 per instruction, both operands K-major
//               from shared memory; tile i accumulates in buffer i mod 2
//   (warps 0 and 1 each walk their loop as a whole warp, with warp-uniform descriptors
//   and coordinates; one elected lane issues every copy, MMA and commit)
//   warps 2-5   epilogue, thread = output row = TMEM lane: 32 columns at a time out of
//               TMEM, bias / GELU / residual in registers, 16-byte stores; it releases an
//               accumulator as soon as it has read it, so a tile's epilogue runs under
//               the next tile's main loop
// Tiles are numbered in groups of kGroupM M-tiles (N-tile-major inside a group): the
// tiles in flight at once share a few row blocks of A and a band of B in L2.
//
// LayerNorm: y = (x - mean) / sqrt(var + eps) * gamma + beta per row, var the biased
// variance, two passes over the row held in registers; 128 threads per row.
#include <cuda_bf16.h>

#include "ra_check.cuh"
#include "ra_internal.h"
#include "ra_layer.h"
#include "ra_ptx.cuh"

namespace ra {

namespace {

constexpr int GM = 128, GN = 256, GK = 64, kStages = 4;
constexpr int kGemmThreads = 192;
constexpr int kAB = GM * GK * 2;            // A box bytes (16 KB)
constexpr int kBB = GN * GK * 2;            // B box bytes (32 KB)
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kStages * kAB;
constexpr int kOffBar = kOffB + kStages * kBB;
constexpr int kNBar = 2 * kStages + 5;      // full[], empty[], acc_full[2], acc_empty[2], drain
constexpr int kGroupM = 32;                 // M-tiles per raster group
constexpr int kOffMisc = kOffBar + kNBar * 8;
constexpr int kGemmSmem = kOffMisc + 16 + 1024;   // + alignment slack
static_assert(kGemmSmem <= 227 * 1024, "shared memory budget");

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void tma_load_2d_w(void* dst, const CUtensorMap* map, uint64_t* bar,
                                              int c0, int c1) {
  asm volatile(
      RA_ELECTED("cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%3, %4}], [%2];") ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ bool wait_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity))
    if (globaltimer_ns() - t0 > limit_ns) return false;
  return true;
}

__device__ __forceinline__ float gelu_exact(float z) {
  return 0.5f * z * (1.0f + erff(z * 0.70710678118654752f));
}

// d GELU / dz = Phi(z) + z phi(z)
__device__ __forceinline__ float gelu_grad(float z) {
  return 0.5f * (1.0f + erff(z * 0.70710678118654752f)) +
         z * 0.39894228040143268f * __expf(-0.5f * z * z);
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4 w, float* f) {
  const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    const float2 p = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wv[x]));
    f[2 * x] = p.x;
    f[2 * x + 1] = p.y;
  }
}

// Output tile of work item `pid`: groups of kGroupM M-tiles, N-tile-major inside a group,
// so that the tiles in flight at once (one per SM) share a few M-tiles of A and a band of
// N-tiles of B in L2.
__device__ __forceinline__ void tile_of(int pid, int mt, int nt, int& tm, int& tn) {
  const int per_group = kGroupM * nt;
  const int first_m = (pid / per_group) * kGroupM;
  const int gsize = (mt - first_m) < kGroupM ? (mt - first_m) : kGroupM;
  const int r = pid % per_group;
  tm = first_m + r % gsize;
  tn = r / gsize;
}

template <int EPI, int A_MN, int B_MN>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const GemmArgs g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = sm + kOffA;
  uint8_t* sB = sm + kOffB;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + kOffBar);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;      // [2]
  uint64_t* acc_empty = acc_full + 2;        // [2]
  uint64_t* drain = acc_empty + 2;
  uint32_t* misc = reinterpret_cast<uint32_t*>(sm + kOffMisc);
  uint32_t* tmem_slot = misc;
  volatile uint32_t* abort_flag = misc + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int mt = g.M / GM, nt = g.N / GN;
  const int ntiles = mt * nt;
  const int nk = g.K / GK;

  if (threadIdx.x == 0) {
    *abort_flag = (*(volatile unsigned int*)g.err != 0u) ? 1u : 0u;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 128);
    }
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (*abort_flag) return;   // an earlier kernel gave up: uniform early exit
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const WaitCtx wc{abort_flag, g.err, g.wait_limit_ns};

  if (warp == 0) {
    // ================================================================ producer =====
    {  // the whole warp; one elected lane issues
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      int it = 0;                               // K steps issued, over all tiles
      bool ok = true;
      for (int pid = blockIdx.x; pid < ntiles && ok; pid += gridDim.x) {
        int tm, tn;
        tile_of(pid, mt, nt, tm, tn);
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % kStages;
          if (it >= kStages && !mbar_wait_w(&empty[s], ((it / kStages) - 1) & 1, wc)) {
            ok = false;
            break;
          }
          mbar_expect_tx_w(&full[s], kAB + kBB);
          // the tile's boxes inside A [M, K] and B [N, K]
          if (!check(g.err, tm >= 0 && (tm + 1) * GM <= g.M && tn >= 0 && (tn + 1) * GN <= g.N &&
                                (kb + 1) * GK <= g.K && s < kStages, kChkTma))
            continue;
          // K-major: one box of rows x 64 K; MN-major: boxes of 64 K rows x 64 M (or N)
          if (A_MN) {
#pragma unroll
            for (int b4 = 0; b4 < GM / 64; ++b4)
              tma_load_2d_w(sA + s * kAB + b4 * 8192, &tmA, &full[s], tm * GM + 64 * b4, kb * GK);
          } else {
            tma_load_2d_w(sA + s * kAB, &tmA, &full[s], kb * GK, tm * GM);
          }
          if (B_MN) {
#pragma unroll
            for (int b4 = 0; b4 < GN / 64; ++b4)
              tma_load_2d_w(sB + s * kBB + b4 * 8192, &tmB, &full[s], tn * GN + 64 * b4, kb * GK);
          } else {
            tma_load_2d_w(sB + s * kBB, &tmB, &full[s], kb * GK, tn * GN);
          }
        }
      }
      if (kChecked && lane == 0) misc[2] = it;                // K steps loaded, compared at the exit
      // let every copy this thread issued land before the CTA can exit
      for (int r = (it > kStages ? it - kStages : 0); r < it; ++r)
        wait_drain(&full[r % kStages], (r / kStages) & 1, g.wait_limit_ns);
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer ===
    {  // the whole warp; one elected lane issues
      constexpr uint32_t idesc = idesc_bf16(GM, GN, A_MN != 0, B_MN != 0);
      const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
      int it = 0, lt = 0;
      bool ok = true;
      for (int pid = blockIdx.x; pid < ntiles && ok; pid += gridDim.x, ++lt) {
        const int buf = lt & 1;
        const uint32_t tacc = tbase + buf * GN;
        if (!check(g.err, buf * GN + GN <= 512, kChkTmem)) { ok = false; break; }
        // the epilogue has read this accumulator's previous tile out of TMEM
        if (lt >= 2 && !mbar_wait_w(&acc_empty[buf], ((lt >> 1) - 1) & 1, wc)) { ok = false; break; }
        tc_fence_after();
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % kStages;
          if (!mbar_wait_w(&full[s], (it / kStages) & 1, wc)) { ok = false; break; }
          tc_fence_after();
          // K-major: +32 bytes per K step of 16; MN-major: +16 rows of 128 bytes, with the
          // 64-wide M (N) blocks 8 KB apart
          const uint64_t ad = A_MN ? sdesc_mnmajor(a0 + s * kAB, 8192) : sdesc_kmajor(a0 + s * kAB);
          const uint64_t bd = B_MN ? sdesc_mnmajor(b0 + s * kBB, 8192) : sdesc_kmajor(b0 + s * kBB);
#pragma unroll
          for (int kk = 0; kk < GK / 16; ++kk)
            umma_ss_w(tacc, ad + (A_MN ? 128 : 2) * kk, bd + (B_MN ? 128 : 2) * kk, idesc,
                    (kb > 0 || kk > 0) ? 1u : 0u);
          umma_commit_w(&empty[s]);
        }
        if (ok) umma_commit_w(&acc_full[buf]);
      }
      if (kChecked && lane == 0) misc[3] = it;                // compared at the exit
      umma_commit_w(drain);
      wait_drain(drain, 0, g.wait_limit_ns);     // every MMA done before TMEM is released
    }
  } else {
    // ================================================================ epilogue =====
    const int q = warp & 3;                       // TMEM lane quadrant of this warp
    const int r = q * 32 + lane;
    int lt = 0;
    for (int pid = blockIdx.x; pid < ntiles; pid += gridDim.x, ++lt) {
      int tm, tn;
      tile_of(pid, mt, nt, tm, tn);
      const int buf = lt & 1;
      const uint32_t trow = tbase + buf * GN + (static_cast<uint32_t>(q * 32) << 16);
      const size_t row = (size_t)tm * GM + r;
      if (!mbar_wait(&acc_full[buf], (lt >> 1) & 1, wc)) break;
      // the output rows and columns of this tile, and its TMEM accumulator
      const bool in_range = check(g.err, row < (size_t)g.M && (size_t)(tn + 1) * GN <= (size_t)g.N &&
                                             tmem_ok(trow, tbase, GN, warp),
                                  kChkGlobal);
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < GN / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(trow + 32 * c, v);
        tmem_wait_ld();
        if (c == GN / 32 - 1) {                   // accumulator fully read: release it
          tc_fence_before();
          mbar_arrive(&acc_empty[buf]);
        }
        if (!in_range) continue;
        const int col = tn * GN + 32 * c;
        const size_t e0 = row * g.N + col;
        float f[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(v[e]);
        if (EPI == kEpiBias || EPI == kEpiBiasGelu || EPI == kEpiBiasResidual ||
            EPI == kEpiBiasGeluZ) {
          const float4* bias4 = reinterpret_cast<const float4*>(g.bias + col);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float4 bb = __ldg(bias4 + e);
            f[4 * e + 0] += bb.x;
            f[4 * e + 1] += bb.y;
            f[4 * e + 2] += bb.z;
            f[4 * e + 3] += bb.w;
          }
        }
        if (EPI == kEpiBiasGeluZ) {                // the pre-activation, as bf16
          uint4* o2 = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(g.out2) + e0);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            o2[e] = make_uint4(pack_bf16x2(f[8 * e], f[8 * e + 1]), pack_bf16x2(f[8 * e + 2], f[8 * e + 3]),
                               pack_bf16x2(f[8 * e + 4], f[8 * e + 5]),
                               pack_bf16x2(f[8 * e + 6], f[8 * e + 7]));
        }
        if (EPI == kEpiBiasGelu || EPI == kEpiBiasGeluZ) {
#pragma unroll
          for (int e = 0; e < 32; ++e) f[e] = gelu_exact(f[e]);
        }
        if (EPI == kEpiBiasResidual || EPI == kEpiGeluGrad) {
          // bf16 [M, N] operand: the residual, or the GELU's input z
          const uint4* aux = reinterpret_cast<const uint4*>(
              reinterpret_cast<const __nv_bfloat16*>(g.aux) + e0);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float z[8];
            bf16x8_to_f32(__ldg(aux + e), z);
#pragma unroll
            for (int x = 0; x < 8; ++x)
              f[8 * e + x] = (EPI == kEpiGeluGrad) ? f[8 * e + x] * gelu_grad(z[x])
                                                   : f[8 * e + x] + z[x];
          }
        }
        if (EPI == kEpiAddF32) {
          // add the fp32 operand and store, 4 columns at a time
          const float4* aux = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(g.aux) + e0);
          float4* o = reinterpret_cast<float4*>(reinterpret_cast<float*>(g.out) + e0);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float4 r4 = __ldg(aux + e);
            o[e] = make_float4(f[4 * e] + r4.x, f[4 * e + 1] + r4.y, f[4 * e + 2] + r4.z,
                               f[4 * e + 3] + r4.w);
          }
        } else if (EPI == kEpiBiasResidual || EPI == kEpiPlainF32) {
          float4* o = reinterpret_cast<float4*>(reinterpret_cast<float*>(g.out) + e0);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            o[e] = make_float4(f[4 * e], f[4 * e + 1], f[4 * e + 2], f[4 * e + 3]);
        } else {
          uint4* o = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(g.out) + e0);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            o[e] = make_uint4(pack_bf16x2(f[8 * e], f[8 * e + 1]), pack_bf16x2(f[8 * e + 2], f[8 * e + 3]),
                              pack_bf16x2(f[8 * e + 4], f[8 * e + 5]),
                              pack_bf16x2(f[8 * e + 6], f[8 * e + 7]));
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (kChecked && threadIdx.x == 0 && !*abort_flag)
    check(g.err, misc[2] == misc[3], kChkSched);   // producer and MMA issuer agree
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// LayerNorm of one row per CTA (128 threads, d / 128 features each, d % 512 == 0 and
// d <= 8192): mean, then the biased variance of the deviations, both reduced in fp32.
template <int OUT_FP32>
__global__ void __launch_bounds__(128)
    layernorm_kernel(const float* __restrict__ x, const float* __restrict__ gamma,
                     const float* __restrict__ beta, float eps, int d, void* out) {
  constexpr int kMaxV = 16;                     // float4 per thread: d <= 16 * 512
  __shared__ float red[2][4];
  const size_t row = blockIdx.x;
  const int nv = d / 512;
  const float4* xr = reinterpret_cast<const float4*>(x + row * d);
  float4 v[kMaxV];
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kMaxV; ++i)
    if (i < nv) {
      v[i] = __ldg(xr + i * 128 + threadIdx.x);
      s += (v[i].x + v[i].y) + (v[i].z + v[i].w);
    }
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) red[0][w] = s;
  __syncthreads();
  const float mean = (red[0][0] + red[0][1] + red[0][2] + red[0][3]) / d;
  float q = 0.f;
#pragma unroll
  for (int i = 0; i < kMaxV; ++i)
    if (i < nv) {
      const float a = v[i].x - mean, b = v[i].y - mean, c = v[i].z - mean, e = v[i].w - mean;
      q += (a * a + b * b) + (c * c + e * e);
    }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
  if (lane == 0) red[1][w] = q;
  __syncthreads();
  const float rstd = rsqrtf((red[1][0] + red[1][1] + red[1][2] + red[1][3]) / d + eps);
#pragma unroll
  for (int i = 0; i < kMaxV; ++i)
    if (i < nv) {
      const int f0 = (i * 128 + threadIdx.x) * 4;
      const float4 gg = __ldg(reinterpret_cast<const float4*>(gamma + f0));
      const float4 bb = __ldg(reinterpret_cast<const float4*>(beta + f0));
      const float y0 = (v[i].x - mean) * rstd * gg.x + bb.x;
      const float y1 = (v[i].y - mean) * rstd * gg.y + bb.y;
      const float y2 = (v[i].z - mean) * rstd * gg.z + bb.z;
      const float y3 = (v[i].w - mean) * rstd * gg.w + bb.w;
      if (OUT_FP32) {
        reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + row * d)[i * 128 + threadIdx.x] =
            make_float4(y0, y1, y2, y3);
      } else {
        reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(out) + row * d)[i * 128 + threadIdx.x] =
            make_uint2(pack_bf16x2(y0, y1), pack_bf16x2(y2, y3));
      }
    }
}

// LayerNorm backward over rows of d features (d % 512 == 0, d <= 4096), kBwdRows rows per
// CTA of 128 threads, each thread owning d / 128 features:
//   yh = (y - mean) * rstd,  dyh = dout * gamma,
//   dy = rstd * (dyh - mean(dyh) - yh * mean(dyh * yh)),
//   dgamma += sum_rows dout * yh,  dbeta += sum_rows dout  (fp32 atomics once per CTA).
// y is the LayerNorm's fp32 input; dout bf16 or fp32; dy written as fp32 and/or bf16.
constexpr int kBwdRows = 16;

template <int DOUT_F32>
__global__ void __launch_bounds__(128)
    layernorm_bwd_kernel(const float* __restrict__ y, const float* __restrict__ gamma,
                         const void* __restrict__ dout, float eps, int d, long long rows,
                         float* dy_f32, __nv_bfloat16* dy_bf16, float* dgamma, float* dbeta) {
  constexpr int kMaxV = 8;
  __shared__ float red[2][4];
  const int nv = d / 512;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float dg[kMaxV][4], db[kMaxV][4];
#pragma unroll
  for (int i = 0; i < kMaxV; ++i)
#pragma unroll
    for (int c = 0; c < 4; ++c) dg[i][c] = db[i][c] = 0.f;
  const long long r0 = (long long)blockIdx.x * kBwdRows;
  for (long long row = r0; row < r0 + kBwdRows && row < rows; ++row) {
    const float4* yr = reinterpret_cast<const float4*>(y + row * d);
    float yv[kMaxV][4], go[kMaxV][4];
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxV; ++i)
      if (i < nv) {
        const float4 t = __ldg(yr + i * 128 + threadIdx.x);
        yv[i][0] = t.x; yv[i][1] = t.y; yv[i][2] = t.z; yv[i][3] = t.w;
        s += (t.x + t.y) + (t.z + t.w);
        const size_t e = (size_t)row * d + (size_t)(i * 128 + threadIdx.x) * 4;
        if (DOUT_F32) {
          const float4 o = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(dout) + e));
          go[i][0] = o.x; go[i][1] = o.y; go[i][2] = o.z; go[i][3] = o.w;
        } else {
          const uint2 o = __ldg(reinterpret_cast<const uint2*>(
              static_cast<const __nv_bfloat16*>(dout) + e));
          const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&o.x));
          const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&o.y));
          go[i][0] = a.x; go[i][1] = a.y; go[i][2] = b.x; go[i][3] = b.y;
        }
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    __syncthreads();                               // red[] reuse across rows
    if (lane == 0) red[0][w] = s;
    __syncthreads();
    const float mean = (red[0][0] + red[0][1] + red[0][2] + red[0][3]) / d;
    float q = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxV; ++i)
      if (i < nv)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float t = yv[i][c] - mean;
          q += t * t;
        }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
    if (lane == 0) red[1][w] = q;
    __syncthreads();
    const float rstd = rsqrtf((red[1][0] + red[1][1] + red[1][2] + red[1][3]) / d + eps);
    float s1 = 0.f, s2 = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxV; ++i)
      if (i < nv) {
        const int f0 = (i * 128 + threadIdx.x) * 4;
        const float4 gg = __ldg(reinterpret_cast<const float4*>(gamma + f0));
        const float gv[4] = {gg.x, gg.y, gg.z, gg.w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float yh = (yv[i][c] - mean) * rstd;
          const float dyh = go[i][c] * gv[c];
          dg[i][c] += go[i][c] * yh;
          db[i][c] += go[i][c];
          yv[i][c] = yh;                          // keep yh, dyh for the last step
          go[i][c] = dyh;
          s1 += dyh;
          s2 += dyh * yh;
        }
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      s1 += __shfl_xor_sync(0xffffffffu, s1, o);
      s2 += __shfl_xor_sync(0xffffffffu, s2, o);
    }
    __syncthreads();
    if (lane == 0) {
      red[0][w] = s1;
      red[1][w] = s2;
    }
    __syncthreads();
    const float m1 = (red[0][0] + red[0][1] + red[0][2] + red[0][3]) / d;
    const float m2 = (red[1][0] + red[1][1] + red[1][2] + red[1][3]) / d;
#pragma unroll
    for (int i = 0; i < kMaxV; ++i)
      if (i < nv) {
        float o[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) o[c] = rstd * (go[i][c] - m1 - yv[i][c] * m2);
        const size_t e = (size_t)row * d + (size_t)(i * 128 + threadIdx.x) * 4;
        if (dy_f32) *reinterpret_cast<float4*>(dy_f32 + e) = make_float4(o[0], o[1], o[2], o[3]);
        if (dy_bf16)
          *reinterpret_cast<uint2*>(dy_bf16 + e) =
              make_uint2(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]));
      }
  }
#pragma unroll
  for (int i = 0; i < kMaxV; ++i)
    if (i < nv)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int f = (i * 128 + threadIdx.x) * 4 + c;
        atomicAdd(dgamma + f, dg[i][c]);
        atomicAdd(dbeta + f, db[i][c]);
      }
}

// out[c] += sum over rows of x[row, c], x bf16 or fp32 [rows, n]; each thread sums 4
// columns over kSumRows rows, then one atomic per column.
constexpr int kSumRows = 256;

template <int X_F32>
__global__ void __launch_bounds__(256)
    colsum_kernel(const void* __restrict__ x, long long rows, int n, float* out) {
  const int c0 = (blockIdx.x * 256 + threadIdx.x) * 4;
  if (c0 >= n) return;
  const long long r0 = (long long)blockIdx.y * kSumRows;
  const long long r1 = r0 + kSumRows < rows ? r0 + kSumRows : rows;
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  for (long long r = r0; r < r1; ++r) {
    const size_t e = (size_t)r * n + c0;
    if (X_F32) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(x) + e));
      a0 += v.x; a1 += v.y; a2 += v.z; a3 += v.w;
    } else {
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(x) + e));
      const float2 p = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
      const float2 q = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
      a0 += p.x; a1 += p.y; a2 += q.x; a3 += q.y;
    }
  }
  atomicAdd(out + c0, a0);
  atomicAdd(out + c0 + 1, a1);
  atomicAdd(out + c0 + 2, a2);
  atomicAdd(out + c0 + 3, a3);
}

}  // namespace

namespace {

template <int EPI, int A_MN, int B_MN>
cudaError_t launch_one(const GemmArgs& g, const CUtensorMap& ta, const CUtensorMap& tb,
                       unsigned grid, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(gemm_kernel<EPI, A_MN, B_MN>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
  if (e != cudaSuccess) return e;
  gemm_kernel<EPI, A_MN, B_MN><<<grid, kGemmThreads, kGemmSmem, s>>>(ta, tb, g);
  return cudaGetLastError();
}

}  // namespace

bool gemm_supported(int epi, int a_mn, int b_mn) {
  if (!a_mn && !b_mn) return epi >= kEpiBias && epi <= kEpiBiasGeluZ;
  if (!a_mn && b_mn)
    return epi == kEpiPlainF32 || epi == kEpiGeluGrad || epi == kEpiAddF32 || epi == kEpiPlainBf16;
  if (a_mn && b_mn) return epi == kEpiPlainF32 || epi == kEpiAddF32;
  return false;
}

cudaError_t launch_gemm(const GemmArgs& g, const CUtensorMap& ta, const CUtensorMap& tb, int epi,
                        int a_mn, int b_mn, cudaStream_t s) {
  if (!gemm_supported(epi, a_mn, b_mn)) return cudaErrorInvalidValue;
  const long long tiles = (long long)(g.M / GM) * (g.N / GN);
  if (tiles <= 0 || tiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  // persistent: one CTA per SM of the current device (shared memory allows one)
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    sms = kAutoSplitSMs;
  const unsigned grid = (unsigned)(tiles < sms ? tiles : sms);
  if (!a_mn && !b_mn) {
    switch (epi) {
      case kEpiBias: return launch_one<kEpiBias, 0, 0>(g, ta, tb, grid, s);
      case kEpiBiasGelu: return launch_one<kEpiBiasGelu, 0, 0>(g, ta, tb, grid, s);
      case kEpiBiasResidual: return launch_one<kEpiBiasResidual, 0, 0>(g, ta, tb, grid, s);
      case kEpiPlainF32: return launch_one<kEpiPlainF32, 0, 0>(g, ta, tb, grid, s);
      case kEpiGeluGrad: return launch_one<kEpiGeluGrad, 0, 0>(g, ta, tb, grid, s);
      case kEpiAddF32: return launch_one<kEpiAddF32, 0, 0>(g, ta, tb, grid, s);
      case kEpiBiasGeluZ: return launch_one<kEpiBiasGeluZ, 0, 0>(g, ta, tb, grid, s);
      default: return launch_one<kEpiPlainBf16, 0, 0>(g, ta, tb, grid, s);
    }
  }
  if (!a_mn) {
    switch (epi) {
      case kEpiPlainF32: return launch_one<kEpiPlainF32, 0, 1>(g, ta, tb, grid, s);
      case kEpiGeluGrad: return launch_one<kEpiGeluGrad, 0, 1>(g, ta, tb, grid, s);
      case kEpiAddF32: return launch_one<kEpiAddF32, 0, 1>(g, ta, tb, grid, s);
      default: return launch_one<kEpiPlainBf16, 0, 1>(g, ta, tb, grid, s);
    }
  }
  if (epi == kEpiAddF32) return launch_one<kEpiAddF32, 1, 1>(g, ta, tb, grid, s);
  return launch_one<kEpiPlainF32, 1, 1>(g, ta, tb, grid, s);
}

cudaError_t launch_layernorm(const float* x, const float* gamma, const float* beta, float eps,
                             long long rows, int d, void* out, int out_fp32, cudaStream_t s) {
  if (d % 512 != 0 || d > 8192 || rows <= 0 || rows > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (out_fp32)
    layernorm_kernel<1><<<(unsigned)rows, 128, 0, s>>>(x, gamma, beta, eps, d, out);
  else
    layernorm_kernel<0><<<(unsigned)rows, 128, 0, s>>>(x, gamma, beta, eps, d, out);
  return cudaGetLastError();
}

cudaError_t launch_layernorm_bwd(const float* y, const float* gamma, const void* dout,
                                 int dout_f32, float eps, long long rows, int d, float* dy_f32,
                                 void* dy_bf16, float* dgamma, float* dbeta, cudaStream_t s) {
  if (d % 512 != 0 || d > 4096 || rows <= 0) return cudaErrorInvalidValue;
  const long long grid = (rows + kBwdRows - 1) / kBwdRows;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  __nv_bfloat16* o16 = static_cast<__nv_bfloat16*>(dy_bf16);
  if (dout_f32)
    layernorm_bwd_kernel<1><<<(unsigned)grid, 128, 0, s>>>(y, gamma, dout, eps, d, rows, dy_f32,
                                                            o16, dgamma, dbeta);
  else
    layernorm_bwd_kernel<0><<<(unsigned)grid, 128, 0, s>>>(y, gamma, dout, eps, d, rows, dy_f32,
                                                            o16, dgamma, dbeta);
  return cudaGetLastError();
}

cudaError_t launch_colsum(const void* x, int x_f32, long long rows, int n, float* out,
                          cudaStream_t s) {
  if (n % 4 != 0 || rows <= 0) return cudaErrorInvalidValue;
  const long long gy = (rows + kSumRows - 1) / kSumRows;
  if (gy > 65535) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)((n / 4 + 255) / 256), (unsigned)gy);
  if (x_f32) colsum_kernel<1><<<grid, 256, 0, s>>>(x, rows, n, out);
  else colsum_kernel<0><<<grid, 256, 0, s>>>(x, rows, n, out);
  return cudaGetLastError();
}

}  // namespace ra
