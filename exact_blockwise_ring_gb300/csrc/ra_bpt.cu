// ra_bpt.cu -- the extern "C" entry points of the blockwise transformer layer: ra_linear,
// ra_layernorm, ra_bpt_workspace_bytes and ra_bpt_fwd (argument checks, workspace layout,
// launch sequence).  The kernels live in ra_gemm.cu and, for the attention, ra_fwd.cu.
#include <cstdarg>
#include <cstdio>

#include "ra_internal.h"
#include "ra_layer.h"

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
                     cudaStream_t st, void* out2 = nullptr) {
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
  g.out2 = out2;
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

// Workspace layout (offsets from the base, each 256-byte aligned).  The forward uses the
// first part; a backward adds the rest (total_train).  The attention region at offset 0 is
// sized for the attention's forward and backward, so both see the same error word.
struct BptWs {
  size_t attn, q, k, v, a, lse, y, h1, f, total;
  size_t z, y2, dy2, dy2f, dy1, da, dxa, dq, dk, dv, total_train;
  int64_t R;
};

bool bpt_layout(const ra_bpt_params_t* p, BptWs* w) {
  const ra_params_t* a = &p->attn;
  size_t attn = ra_fwd_workspace_bytes(a);
  if (attn == 0) return false;
  const size_t attn_b = ra_bwd_workspace_bytes(a);
  if (attn_b > attn) attn = attn_b;
  const int64_t rows = (int64_t)a->batch * a->seq_len;
  const int64_t d = (int64_t)a->heads * a->head_dim;
  const int64_t dkv = (int64_t)(a->kv_heads > 0 ? a->kv_heads : a->heads) * a->head_dim;
  int64_t R = p->block_rows > 0 ? p->block_rows : (rows < 16384 ? rows : 16384);
  if (R > rows) R = rows;
  w->R = R;
  size_t off = r256(attn);
  w->attn = 0;
  w->q = off; off += r256((size_t)rows * d * 2);
  w->k = off; off += r256((size_t)rows * dkv * 2);
  w->v = off; off += r256((size_t)rows * dkv * 2);
  w->a = off; off += r256((size_t)rows * d * 2);
  w->lse = off; off += r256((size_t)a->batch * a->heads * a->seq_len * 4);
  w->y = off; off += r256((size_t)R * d * 4);
  w->h1 = off; off += r256((size_t)R * d * 2);
  w->f = off; off += r256((size_t)R * p->d_ff * 2);
  w->total = off;
  w->z = off; off += r256((size_t)R * p->d_ff * 2);
  w->y2 = off; off += r256((size_t)R * d * 4);
  w->dy2 = off; off += r256((size_t)R * d * 2);
  w->dy2f = off; off += r256((size_t)R * d * 4);
  w->dy1 = off; off += r256((size_t)R * d * 2);
  w->da = off; off += r256((size_t)rows * d * 2);
  w->dxa = off; off += r256((size_t)rows * d * 4);
  w->dq = off; off += r256((size_t)rows * d * 2);
  w->dk = off; off += r256((size_t)rows * dkv * 2);
  w->dv = off; off += r256((size_t)rows * dkv * 2);
  w->total_train = off;
  return true;
}

ra_status_t cuda_err(cudaError_t e, const char* what) {
  return e == cudaSuccess ? RA_OK : bfail(RA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

ra_status_t check_bpt(const ra_bpt_params_t* p) {
  if (!p) return bfail(RA_ERR_INVALID_ARG, "params is NULL");
  const ra_params_t* a = &p->attn;
  if (ra_fwd_workspace_bytes(a) == 0)
    return bfail(RA_ERR_INVALID_ARG, "invalid attention parameters (see ra_fwd)");
  const long long dkv = (long long)(a->kv_heads > 0 ? a->kv_heads : a->heads) * a->head_dim;
  if (dkv % 256 != 0)
    return bfail(RA_ERR_UNSUPPORTED, "kv_heads * head_dim (%lld) must be a multiple of 256", dkv);
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

  // projections over the whole sequence: [B*L, d] rows are [B, L, H, D] tensors (K and V
  // [B, L, H_kv, D])
  const int dkv = (a->kv_heads > 0 ? a->kv_heads : a->heads) * a->head_dim;
  if ((s = run_linear(rows, d, d, x, wt->wq, wt->bq, nullptr, RA_EPI_BIAS, Q, err, st)) != RA_OK ||
      (s = run_linear(rows, d, dkv, x, wt->wk, wt->bk, nullptr, RA_EPI_BIAS, K, err, st)) != RA_OK ||
      (s = run_linear(rows, d, dkv, x, wt->wv, wt->bv, nullptr, RA_EPI_BIAS, V, err, st)) != RA_OK)
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

size_t ra_bpt_train_workspace_bytes(const ra_bpt_params_t* p) {
  if (check_bpt(p) != RA_OK) return 0;
  if ((long long)p->attn.heads * p->attn.head_dim > 4096) return 0;
  BptWs w;
  return bpt_layout(p, &w) ? w.total_train : 0;
}

ra_status_t ra_bpt_bwd(const ra_bpt_params_t* p, const void* x, const ra_bpt_weights_t* wt,
                       const void* dout, const ra_bpt_grads_t* gr, void* workspace,
                       size_t workspace_bytes, void* stream) {
  ra_status_t s = check_bpt(p);
  if (s != RA_OK) return s;
  if ((long long)p->attn.heads * p->attn.head_dim > 4096)
    return bfail(RA_ERR_UNSUPPORTED, "the layer's backward needs d_model <= 4096");
  if (!x || !wt || !dout || !gr) return bfail(RA_ERR_INVALID_ARG, "null pointer");
  const void* ptrs[] = {wt->wq, wt->wk, wt->wv, wt->wo, wt->w1, wt->w2, wt->bq, wt->bk,
                        wt->bv, wt->bo, wt->b1, wt->b2, wt->ln1_g, wt->ln1_b, wt->ln2_g,
                        wt->ln2_b, x, dout, gr->dx, gr->wq, gr->wk, gr->wv, gr->wo, gr->w1,
                        gr->w2, gr->bq, gr->bk, gr->bv, gr->bo, gr->b1, gr->b2, gr->ln1_g,
                        gr->ln1_b, gr->ln2_g, gr->ln2_b};
  for (const void* q : ptrs) {
    if (!q) return bfail(RA_ERR_INVALID_ARG, "null weight, gradient or tensor pointer");
    if (!al16(q)) return bfail(RA_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  }
  BptWs w;
  if (!bpt_layout(p, &w)) return bfail(RA_ERR_INVALID_ARG, "invalid parameters");
  if (!workspace || workspace_bytes < w.total_train || !al16(workspace))
    return bfail(RA_ERR_WORKSPACE, "workspace needs %zu bytes (16-byte aligned), got %zu",
                 w.total_train, workspace_bytes);
  const ra_params_t* a = &p->attn;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  unsigned int* err = reinterpret_cast<unsigned int*>(ws);
  const int64_t rows = (int64_t)a->batch * a->seq_len;
  const int d = a->heads * a->head_dim;
  const int d_ff = p->d_ff;
  const int dkv = (a->kv_heads > 0 ? a->kv_heads : a->heads) * a->head_dim;
  const float eps = p->ln_eps > 0.f ? p->ln_eps : 1e-5f;
  const uint8_t* xb = static_cast<const uint8_t*>(x);
  const uint8_t* dob = static_cast<const uint8_t*>(dout);
  uint8_t *Q = ws + w.q, *K = ws + w.k, *V = ws + w.v, *A = ws + w.a;
  float* lse = reinterpret_cast<float*>(ws + w.lse);
  float* Y = reinterpret_cast<float*>(ws + w.y);
  float* Y2 = reinterpret_cast<float*>(ws + w.y2);
  float* DY2F = reinterpret_cast<float*>(ws + w.dy2f);
  float* DXA = reinterpret_cast<float*>(ws + w.dxa);
  void *H1 = ws + w.h1, *F = ws + w.f, *Z = ws + w.z, *DY2 = ws + w.dy2, *DY1 = ws + w.dy1;
  uint8_t *DA = ws + w.da, *DQ = ws + w.dq, *DK = ws + w.dk, *DV = ws + w.dv;

  // gradients accumulated over blocks start at zero
  struct { float* p; size_t n; } acc[] = {
      {gr->wo, (size_t)d * d}, {gr->w1, (size_t)d_ff * d}, {gr->w2, (size_t)d * d_ff},
      {gr->bq, (size_t)d}, {gr->bk, (size_t)dkv}, {gr->bv, (size_t)dkv}, {gr->bo, (size_t)d},
      {gr->b1, (size_t)d_ff}, {gr->b2, (size_t)d}, {gr->ln1_g, (size_t)d},
      {gr->ln1_b, (size_t)d}, {gr->ln2_g, (size_t)d}, {gr->ln2_b, (size_t)d}};
  for (auto& z : acc)
    if ((s = cuda_err(cudaMemsetAsync(z.p, 0, z.n * 4, st), "cudaMemsetAsync(gradient)")) != RA_OK)
      return s;

  for (int64_t r0 = 0; r0 < rows; r0 += w.R) {
    const int64_t R = (rows - r0) < w.R ? (rows - r0) : w.R;
    const size_t o16 = (size_t)r0 * d * 2;
    // recompute the block's forward: y1, h1 = LN1(y1), z, f = GELU(z), y2
    if ((s = run_linear(R, d, d, A + o16, wt->wo, wt->bo, xb + o16, kEpiBiasResidual, Y, err,
                        st)) != RA_OK)
      return s;
    if ((s = cuda_err(launch_layernorm(Y, wt->ln1_g, wt->ln1_b, eps, R, d, H1, 0, st),
                      "LayerNorm launch")) != RA_OK)
      return s;
    // f = GELU(z) exactly as the forward rounded it, and z itself for GELU'
    if ((s = run_gemm(R, d_ff, d, H1, 0, wt->w1, 0, wt->b1, nullptr, kEpiBiasGeluZ, F, err, st,
                      Z)) != RA_OK)
      return s;
    if ((s = run_linear(R, d_ff, d, F, wt->w2, wt->b2, H1, kEpiBiasResidual, Y2, err, st)) != RA_OK)
      return s;
    // LN2 backward: dy2 (fp32 and bf16), dgamma2, dbeta2
    if ((s = cuda_err(launch_layernorm_bwd(Y2, wt->ln2_g, dob + o16, 0, eps, R, d, DY2F, DY2,
                                           gr->ln2_g, gr->ln2_b, st),
                      "LayerNorm backward launch")) != RA_OK)
      return s;
    // W2: dW2 += dy2^T f, db2 += sum dy2, dz = (dy2 W2) * GELU'(z) (over z, in place)
    if ((s = run_gemm(d, d_ff, (int)R, DY2, 1, F, 1, nullptr, gr->w2, kEpiAddF32, gr->w2, err,
                      st)) != RA_OK ||
        (s = cuda_err(launch_colsum(DY2F, 1, R, d, gr->b2, st), "column sum")) != RA_OK ||
        (s = run_gemm(R, d_ff, d, DY2, 0, wt->w2, 1, nullptr, Z, kEpiGeluGrad, Z, err, st)) != RA_OK)
      return s;
    // W1: dW1 += dz^T h1, db1 += sum dz, dh1 = dz W1 + dy2 (into the y2 buffer)
    if ((s = run_gemm(d_ff, d, (int)R, Z, 1, H1, 1, nullptr, gr->w1, kEpiAddF32, gr->w1, err,
                      st)) != RA_OK ||
        (s = cuda_err(launch_colsum(Z, 0, R, d_ff, gr->b1, st), "column sum")) != RA_OK ||
        (s = run_gemm(R, d, d_ff, Z, 0, wt->w1, 1, nullptr, DY2F, kEpiAddF32, Y2, err, st)) != RA_OK)
      return s;
    // LN1 backward: dy1 into the dx accumulator (the residual path) and as bf16
    float* dxa_blk = DXA + (size_t)r0 * d;
    if ((s = cuda_err(launch_layernorm_bwd(Y, wt->ln1_g, Y2, 1, eps, R, d, dxa_blk, DY1,
                                           gr->ln1_g, gr->ln1_b, st),
                      "LayerNorm backward launch")) != RA_OK)
      return s;
    // Wo: dWo += dy1^T a, dbo += sum dy1, da = dy1 Wo
    if ((s = run_gemm(d, d, (int)R, DY1, 1, A + o16, 1, nullptr, gr->wo, kEpiAddF32, gr->wo, err,
                      st)) != RA_OK ||
        (s = cuda_err(launch_colsum(dxa_blk, 1, R, d, gr->bo, st), "column sum")) != RA_OK ||
        (s = run_gemm(R, d, d, DY1, 0, wt->wo, 1, nullptr, nullptr, kEpiPlainBf16, DA + o16, err,
                      st)) != RA_OK)
      return s;
  }
  // the attention's backward over the whole sequence (its workspace is the first region)
  if ((s = ra_bwd(a, Q, K, V, A, RA_BF16, lse, DA, DQ, DK, DV, ws + w.attn, w.q, stream)) !=
      RA_OK)
    return s;
  // projections: dx += dQ Wq + dK Wk + dV Wv; dW = d(Q|K|V)^T x; db = column sums
  const void* dqkv[3] = {DQ, DK, DV};
  const void* wqkv[3] = {wt->wq, wt->wk, wt->wv};
  float* gw[3] = {gr->wq, gr->wk, gr->wv};
  float* gb[3] = {gr->bq, gr->bk, gr->bv};
  for (int t = 0; t < 3; ++t) {
    const int n_out = t == 0 ? d : dkv;          // Q is d wide, K and V H_kv * D
    if ((s = run_gemm(rows, d, n_out, dqkv[t], 0, wqkv[t], 1, nullptr, DXA, kEpiAddF32, DXA, err,
                      st)) != RA_OK ||
        (s = run_gemm(n_out, d, (int)rows, dqkv[t], 1, x, 1, nullptr, nullptr, kEpiPlainF32,
                      gw[t], err, st)) != RA_OK ||
        (s = cuda_err(launch_colsum(dqkv[t], 0, rows, n_out, gb[t], st), "column sum")) != RA_OK)
      return s;
  }
  return cuda_err(launch_dq_convert(DXA, gr->dx, 1.0f, (size_t)rows * d, st), "dx convert");
}

}  // extern "C"
