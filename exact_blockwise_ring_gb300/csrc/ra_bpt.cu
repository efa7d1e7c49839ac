// ra_bpt.cu -- the extern "C" entry points of the blockwise transformer layer: ra_linear,
// ra_layernorm, ra_bpt_workspace_bytes and ra_bpt_fwd (argument checks, workspace layout,
// launch sequence).  The kernels live in ra_gemm.cu and, for the attention, ra_fwd.cu.
#include <cstdarg>
#include <cstdio>

#include "ra_internal.h"

namespace ra {
namespace {

ra_status_t bfail(ra_status_t s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  set_last_error_message(buf);
  return s;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t r256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Shape and pointer checks of one Linear call; pointers may be checked by the caller.
ra_status_t check_linear(int64_t rows, int in_f, int out_f, int epi) {
  if (rows < 1 || in_f < 1 || out_f < 1)
    return bfail(RA_ERR_INVALID_ARG, "rows, in_features and out_features must be >= 1");
  if (epi < RA_EPI_BIAS || epi > RA_EPI_BIAS_RESIDUAL)
    return bfail(RA_ERR_INVALID_ARG, "epilogue must be an ra_epilogue_t value");
  if (rows % 128 || out_f % 256 || in_f % 64)
    return bfail(RA_ERR_UNSUPPORTED,
                 "ra_linear needs rows %% 128 == 0, out_features %% 256 == 0, in_features %% 64 "
                 "== 0 (got %lld, %d, %d)", (long long)rows, out_f, in_f);
  if (rows > (1LL << 31) - 1 || (long long)rows * out_f > (1LL << 40))
    return bfail(RA_ERR_INVALID_ARG, "tensor too large");
  return RA_OK;
}

// out[M, N] = epilogue(A B): A stored [M, K] (a_mn = 0) or [K, M] (a_mn = 1), B stored
// [N, K] (b_mn = 0) or [K, N] (b_mn = 1); shapes already checked.
ra_status_t run_gemm(int64_t M, int N, int K, const void* a, int a_mn, const void* b, int b_mn,
                     const float* bias, const void* aux, int epi, void* out, unsigned int* err,
                     cudaStream_t st) {
  CUtensorMap ta, tb;
  ra_status_t s;
  if (a_mn) s = encode_2d_bf16(&ta, a, M, K, 64, 64);
  else s = encode_2d_bf16(&ta, a, K, M, 64, 128);
  if (s != RA_OK) return s;
  if (b_mn) s = encode_2d_bf16(&tb, b, N, K, 64, 64);
  else s = encode_2d_bf16(&tb, b, K, N, 64, 256);
  if (s != RA_OK) return s;
  GemmArgs g{};
  g.M = (int)M;
  g.N = N;
  g.K = K;
  g.bias = bias;
  g.aux = aux;
  g.out = out;
  g.err = err;
  g.wait_limit_ns = kWaitLimitNs;
  cudaError_t e = launch_gemm(g, ta, tb, epi, a_mn, b_mn, st);
  if (e != cudaSuccess) return bfail(RA_ERR_CUDA, "GEMM launch: %s", cudaGetErrorString(e));
  return RA_OK;
}

// y = x W^T + b (and its fused epilogue): A = x [rows, in], B = W [out, in], both K-major.
ra_status_t run_linear(int64_t rows, int in_f, int out_f, const void* x, const void* weight,
                       const float* bias, const void* residual, int epi, void* out,
                       unsigned int* err, cudaStream_t st) {
  return run_gemm(rows, out_f, in_f, x, 0, weight, 0, bias, residual, epi, out, err, st);
}

// Workspace layout of ra_bpt_fwd (offsets from the base, each 256-byte aligned).
struct BptWs {
  size_t attn, q, k, v, a, lse, y, h1, f, total;
  int64_t R;
};

bool bpt_layout(const ra_bpt_params_t* p, BptWs* w) {
  const ra_params_t* a = &p->attn;
  const size_t attn = ra_fwd_workspace_bytes(a);
  if (attn == 0) return false;
  const int64_t rows = (int64_t)a->batch * a->seq_len;
  const int64_t d = (int64_t)a->heads * a->head_dim;
  int64_t R = p->block_rows > 0 ? p->block_rows : (rows < 16384 ? rows : 16384);
  if (R > rows) R = rows;
  w->R = R;
  size_t off = r256(attn);
  w->attn = 0;
  w->q = off; off += r256((size_t)rows * d * 2);
  w->k = off; off += r256((size_t)rows * d * 2);
  w->v = off; off += r256((size_t)rows * d * 2);
  w->a = off; off += r256((size_t)rows * d * 2);
  w->lse = off; off += r256((size_t)a->batch * a->heads * a->seq_len * 4);
  w->y = off; off += r256((size_t)R * d * 4);
  w->h1 = off; off += r256((size_t)R * d * 2);
  w->f = off; off += r256((size_t)R * p->d_ff * 2);
  w->total = off;
  return true;
}

ra_status_t check_bpt(const ra_bpt_params_t* p) {
  if (!p) return bfail(RA_ERR_INVALID_ARG, "params is NULL");
  const ra_params_t* a = &p->attn;
  if (a->kv_heads != 0 && a->kv_heads != a->heads)
    return bfail(RA_ERR_INVALID_ARG, "the layer projects K and V to all heads: kv_heads must be 0");
  if (ra_fwd_workspace_bytes(a) == 0)
    return bfail(RA_ERR_INVALID_ARG, "invalid attention parameters (see ra_fwd)");
  const long long d = (long long)a->heads * a->head_dim;
  if (d % 512 != 0 || d > 8192)
    return bfail(RA_ERR_UNSUPPORTED, "d_model = heads * head_dim (%lld) must be a multiple of 512 "
                 "and at most 8192", d);
  if (p->d_ff < 256 || p->d_ff % 256 != 0)
    return bfail(RA_ERR_UNSUPPORTED, "d_ff (%d) must be a positive multiple of 256", p->d_ff);
  if (p->block_rows < 0 || p->block_rows % 128 != 0)
    return bfail(RA_ERR_INVALID_ARG, "block_rows must be 0 or a positive multiple of 128");
  if (!(p->ln_eps >= 0.f))
    return bfail(RA_ERR_INVALID_ARG, "ln_eps must be >= 0");
  return RA_OK;
}

}  // namespace
}  // namespace ra

using namespace ra;

extern "C" {

ra_status_t ra_linear(int64_t rows, int in_features, int out_features, const void* x,
                      const void* weight, const float* bias, const void* residual, int epilogue,
                      void* out, void* workspace, size_t workspace_bytes, void* stream) {
  ra_status_t s = check_linear(rows, in_features, out_features, epilogue);
  if (s != RA_OK) return s;
  if (!x || !weight || !bias || !out || (epilogue == RA_EPI_BIAS_RESIDUAL && !residual))
    return bfail(RA_ERR_INVALID_ARG, "null tensor pointer");
  if (!al16(x) || !al16(weight) || !al16(bias) || !al16(out) || (residual && !al16(residual)))
    return bfail(RA_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (!workspace || workspace_bytes < kWsHeader || !al16(workspace))
    return bfail(RA_ERR_WORKSPACE, "workspace needs %zu bytes (16-byte aligned)", kWsHeader);
  return run_linear(rows, in_features, out_features, x, weight, bias, residual, epilogue, out,
                    static_cast<unsigned int*>(workspace), reinterpret_cast<cudaStream_t>(stream));
}

ra_status_t ra_layernorm(int64_t rows, int features, const float* x, const float* gamma,
                         const float* beta, float eps, void* out, int out_dtype, void* stream) {
  if (rows < 1 || features < 1) return bfail(RA_ERR_INVALID_ARG, "rows and features must be >= 1");
  if (features % 512 != 0 || features > 8192)
    return bfail(RA_ERR_UNSUPPORTED, "features (%d) must be a multiple of 512 and <= 8192",
                 features);
  if (rows > (1LL << 31) - 1) return bfail(RA_ERR_INVALID_ARG, "too many rows");
  if (!(eps > 0.f)) return bfail(RA_ERR_INVALID_ARG, "eps must be > 0");
  if (out_dtype != RA_BF16 && out_dtype != RA_FP32)
    return bfail(RA_ERR_INVALID_ARG, "out_dtype must be RA_BF16 or RA_FP32");
  if (!x || !gamma || !beta || !out) return bfail(RA_ERR_INVALID_ARG, "null tensor pointer");
  if (!al16(x) || !al16(gamma) || !al16(beta) || !al16(out))
    return bfail(RA_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  cudaError_t e = launch_layernorm(x, gamma, beta, eps, rows, features, out, out_dtype == RA_FP32,
                                   reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return bfail(RA_ERR_CUDA, "LayerNorm launch: %s", cudaGetErrorString(e));
  return RA_OK;
}

size_t ra_bpt_workspace_bytes(const ra_bpt_params_t* p) {
  if (check_bpt(p) != RA_OK) return 0;
  BptWs w;
  return bpt_layout(p, &w) ? w.total : 0;
}

ra_status_t ra_bpt_fwd(const ra_bpt_params_t* p, const void* x, const ra_bpt_weights_t* wt,
                       void* out, int out_dtype, void* workspace, size_t workspace_bytes,
                       void* stream) {
  ra_status_t s = check_bpt(p);
  if (s != RA_OK) return s;
  if (!x || !wt || !out) return bfail(RA_ERR_INVALID_ARG, "null pointer");
  const void* ptrs[] = {wt->wq, wt->wk, wt->wv, wt->wo, wt->w1, wt->w2, wt->bq, wt->bk,
                        wt->bv, wt->bo, wt->b1, wt->b2, wt->ln1_g, wt->ln1_b, wt->ln2_g,
                        wt->ln2_b, x, out};
  for (const void* q : ptrs) {
    if (!q) return bfail(RA_ERR_INVALID_ARG, "null weight or tensor pointer");
    if (!al16(q)) return bfail(RA_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  }
  if (out_dtype != RA_BF16 && out_dtype != RA_FP32)
    return bfail(RA_ERR_INVALID_ARG, "out_dtype must be RA_BF16 or RA_FP32");
  BptWs w;
  if (!bpt_layout(p, &w)) return bfail(RA_ERR_INVALID_ARG, "invalid parameters");
  if (!workspace || workspace_bytes < w.total || !al16(workspace))
    return bfail(RA_ERR_WORKSPACE, "workspace needs %zu bytes (16-byte aligned), got %zu", w.total,
                 workspace_bytes);
  const ra_params_t* a = &p->attn;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  unsigned int* err = reinterpret_cast<unsigned int*>(ws);   // the attention's error word
  const int64_t rows = (int64_t)a->batch * a->seq_len;
  const int d = a->heads * a->head_dim;
  const int d_ff = p->d_ff;
  const float eps = p->ln_eps > 0.f ? p->ln_eps : 1e-5f;
  void *Q = ws + w.q, *K = ws + w.k, *V = ws + w.v, *A = ws + w.a;
  float* lse = reinterpret_cast<float*>(ws + w.lse);
  float* Y = reinterpret_cast<float*>(ws + w.y);
  void *H1 = ws + w.h1, *F = ws + w.f;

  // projections over the whole sequence: [B*L, d] rows are [B, L, H, D] tensors
  if ((s = run_linear(rows, d, d, x, wt->wq, wt->bq, nullptr, RA_EPI_BIAS, Q, err, st)) != RA_OK ||
      (s = run_linear(rows, d, d, x, wt->wk, wt->bk, nullptr, RA_EPI_BIAS, K, err, st)) != RA_OK ||
      (s = run_linear(rows, d, d, x, wt->wv, wt->bv, nullptr, RA_EPI_BIAS, V, err, st)) != RA_OK)
    return s;
  // ring attention; its workspace is the first part of this one (same error word)
  if ((s = ra_fwd(a, Q, K, V, A, RA_BF16, lse, nullptr, ws + w.attn, w.q, stream)) != RA_OK)
    return s;
  // per block of rows: Wo + residual, LN1, W1 + GELU, W2 + residual, LN2
  const uint8_t* xb = static_cast<const uint8_t*>(x);
  const uint8_t* ab = static_cast<const uint8_t*>(A);
  uint8_t* ob = static_cast<uint8_t*>(out);
  const size_t osz = out_dtype == RA_FP32 ? 4 : 2;
  for (int64_t r0 = 0; r0 < rows; r0 += w.R) {
    const int64_t R = (rows - r0) < w.R ? (rows - r0) : w.R;
    const size_t o16 = (size_t)r0 * d * 2;
    if ((s = run_linear(R, d, d, ab + o16, wt->wo, wt->bo, xb + o16, RA_EPI_BIAS_RESIDUAL, Y, err,
                        st)) != RA_OK)
      return s;
    cudaError_t e = launch_layernorm(Y, wt->ln1_g, wt->ln1_b, eps, R, d, H1, 0, st);
    if (e != cudaSuccess) return bfail(RA_ERR_CUDA, "LayerNorm launch: %s", cudaGetErrorString(e));
    if ((s = run_linear(R, d, d_ff, H1, wt->w1, wt->b1, nullptr, RA_EPI_BIAS_GELU, F, err,
                        st)) != RA_OK ||
        (s = run_linear(R, d_ff, d, F, wt->w2, wt->b2, H1, RA_EPI_BIAS_RESIDUAL, Y, err, st)) !=
            RA_OK)
      return s;
    e = launch_layernorm(Y, wt->ln2_g, wt->ln2_b, eps, R, d, ob + (size_t)r0 * d * osz,
                         out_dtype == RA_FP32, st);
    if (e != cudaSuccess) return bfail(RA_ERR_CUDA, "LayerNorm launch: %s", cudaGetErrorString(e));
  }
  return RA_OK;
}

}  // extern "C"
