// ra_layer.h -- declarations shared by the blockwise transformer layer's kernels
// (ra_gemm.cu) and entry points (ra_bpt.cu); kept apart from ra_internal.h, which the
// attention kernels include.
#pragma once

#include "ra_internal.h"

namespace ra {

// Dense kernels of the blockwise transformer layer (ra_gemm.cu).
// Epilogues (out[M, N] from the fp32 accumulator acc):
//   kEpiBias          bf16  acc + bias
//   kEpiBiasGelu      bf16  GELU(acc + bias)
//   kEpiBiasResidual  fp32  acc + bias + aux (bf16 [M, N])
//   kEpiPlainF32      fp32  acc
//   kEpiGeluGrad      bf16  acc * GELU'(aux), aux = the GELU's input z (bf16 [M, N])
//   kEpiAddF32        fp32  acc + aux (fp32 [M, N])
//   kEpiPlainBf16     bf16  acc
//   kEpiBiasGeluZ     bf16  GELU(acc + bias), and bf16 acc + bias into out2 (the same fp32
//                     value rounded before and after GELU, as the forward rounds it)
enum GemmEpilogue : int {
  kEpiBias = 0, kEpiBiasGelu = 1, kEpiBiasResidual = 2, kEpiPlainF32 = 3, kEpiGeluGrad = 4,
  kEpiAddF32 = 5, kEpiPlainBf16 = 6, kEpiBiasGeluZ = 7
};

// out[M, N] = epilogue(sum_k A[m, k] B[n, k]); M % 128, N % 256, K % 64 == 0.  A is read
// K-major (stored [M, K]) or, with a_mn, MN-major (stored [K, M]); B likewise ([N, K] or
// [K, N]).  Supported: (a_mn, b_mn) = (0, 0) with every epilogue, (0, 1) with kEpiPlainF32,
// kEpiGeluGrad, kEpiAddF32, kEpiPlainBf16, and (1, 1) with kEpiPlainF32.
struct GemmArgs {
  int M, N, K;
  const float* bias;        // [N] fp32 (kEpiBias*, the GELU ones, kEpiBiasResidual)
  const void* aux;          // [M, N] operand of kEpiBiasResidual, kEpiGeluGrad, kEpiAddF32
  void* out;
  void* out2;               // [M, N] second output of kEpiBiasGeluZ
  unsigned int* err;        // workspace error word
  uint64_t wait_limit_ns;
};

bool gemm_supported(int epi, int a_mn, int b_mn);
cudaError_t launch_gemm(const GemmArgs& g, const CUtensorMap& ta, const CUtensorMap& tb, int epi,
                        int a_mn, int b_mn, cudaStream_t s);
cudaError_t launch_layernorm(const float* x, const float* gamma, const float* beta, float eps,
                             long long rows, int d, void* out, int out_fp32, cudaStream_t s);
cudaError_t launch_layernorm_bwd(const float* y, const float* gamma, const void* dout,
                                 int dout_f32, float eps, long long rows, int d, float* dy_f32,
                                 void* dy_bf16, float* dgamma, float* dbeta, cudaStream_t s);
cudaError_t launch_colsum(const void* x, int x_f32, long long rows, int n, float* out,
                          cudaStream_t s);


// A 2-D bf16 [outer, inner] row-major tensor map with 128-byte swizzled boxes of
// box_outer rows x box_inner elements (ra_api.cu).
ra_status_t encode_2d_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                           uint32_t box_inner, uint32_t box_outer);

}  // namespace ra
