// ra_api.cu -- the extern "C" boundary of libra: argument validation, workspace layout,
// TMA tensor-map encoding, kernel launches, error reporting and the host work model.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "ra_check.cuh"
#include "ra_internal.h"
#include "ra_layer.h"

namespace ra {
namespace {

thread_local char g_msg[512] = "";

ra_status_t fail(ra_status_t s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return s;
}

ra_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(RA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---- validation -------------------------------------------------------------------
ra_status_t check_params(const ra_params_t* p, bool gpu_shapes) {
  if (!p) return fail(RA_ERR_INVALID_ARG, "params is NULL");
  if (p->batch < 1 || p->heads < 1 || p->seq_len < 1 || p->P < 1)
    return fail(RA_ERR_INVALID_ARG, "batch, heads, seq_len and P must be >= 1");
  if (p->P > 1024) return fail(RA_ERR_INVALID_ARG, "P must be <= 1024");
  if (p->block < 1) return fail(RA_ERR_INVALID_ARG, "block must be >= 1");
  if (p->layout != RA_LAYOUT_CONTIGUOUS && p->layout != RA_LAYOUT_STRIPED &&
      p->layout != RA_LAYOUT_ZIGZAG)
    return fail(RA_ERR_INVALID_ARG,
                "layout must be RA_LAYOUT_CONTIGUOUS, RA_LAYOUT_STRIPED or RA_LAYOUT_ZIGZAG");
  if (p->causal != 0 && p->causal != 1) return fail(RA_ERR_INVALID_ARG, "causal must be 0 or 1");
  if (p->kv_heads < 0 || (p->kv_heads > 0 && p->heads % p->kv_heads != 0))
    return fail(RA_ERR_INVALID_ARG, "kv_heads (%d) must be 0 or a divisor of heads (%d)",
                p->kv_heads, p->heads);
  if (p->seq_len % p->P != 0 || (p->seq_len / p->P) % p->block != 0)
    return fail(RA_ERR_INVALID_ARG, "seq_len (%lld) must be divisible by P * block (%d * %d)",
                (long long)p->seq_len, p->P, p->block);
  if (p->layout == RA_LAYOUT_ZIGZAG && (p->seq_len / p->P) % (2LL * p->block) != 0)
    return fail(RA_ERR_INVALID_ARG,
                "zigzag: seq_len (%lld) must be divisible by 2 * P * block (2 * %d * %d)",
                (long long)p->seq_len, p->P, p->block);
  if (!gpu_shapes) return RA_OK;
  if (p->head_dim < 1) return fail(RA_ERR_INVALID_ARG, "head_dim must be >= 1");
  if (p->head_dim != 64 && p->head_dim != 128)
    return fail(RA_ERR_UNSUPPORTED, "head_dim %d: kernels exist for 64 and 128", p->head_dim);
  if (p->block != 128 && p->block != 256)
    return fail(RA_ERR_UNSUPPORTED, "block %d: kernels exist for 128 and 256", p->block);
  if (!(p->softmax_scale >= 0.f) || !std::isfinite(p->softmax_scale))
    return fail(RA_ERR_INVALID_ARG, "softmax_scale must be finite and >= 0");
  if (p->n_split < 0 || (p->n_split > 0 && p->P % p->n_split != 0))
    return fail(RA_ERR_INVALID_ARG, "n_split must be 0 or a divisor of P");
  const long long elems = (long long)p->batch * p->seq_len * p->heads * p->head_dim;
  if (elems <= 0 || elems > (1LL << 40))
    return fail(RA_ERR_INVALID_ARG, "tensor too large");
  const long long bhl = (long long)p->batch * p->heads * p->seq_len;
  if (bhl > (1LL << 36)) return fail(RA_ERR_INVALID_ARG, "tensor too large");
  return RA_OK;
}

int kv_of(const ra_params_t* p) { return p->kv_heads > 0 ? p->kv_heads : p->heads; }

float scale_of(const ra_params_t* p) {
  return p->softmax_scale > 0.f ? p->softmax_scale : 1.0f / std::sqrt((float)p->head_dim);
}

int npair_of(const ra_params_t* p) {
  const int T = (int)(p->seq_len / p->P / kTile);
  return (T + 1) / 2;
}

int n_split_of(const ra_params_t* p) {
  if (p->n_split > 0) return p->n_split;
  const long long ctas = (long long)p->batch * p->heads * p->P * npair_of(p);
  if (ctas >= kAutoSplitSMs) return 1;
  int best = 1;
  for (int g = 1; g <= p->P; ++g)
    if (p->P % g == 0 && ctas * g <= 2LL * kAutoSplitSMs) best = g;
  return best;
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

size_t fwd_ws(const ra_params_t* p) {
  const int g = n_split_of(p);
  size_t bytes = kWsHeader;
  if (g > 1) {
    const size_t o = (size_t)p->batch * p->seq_len * p->heads * p->head_dim * 4;
    const size_t l = (size_t)p->batch * p->heads * p->seq_len * 4;
    bytes += round256(g * o) + round256(g * l);
  }
  return bytes;
}

size_t bwd_ws(const ra_params_t* p) {
  const size_t o = (size_t)p->batch * p->seq_len * p->heads * p->head_dim * 4;
  const size_t l = (size_t)p->batch * p->heads * p->seq_len * 4;
  return kWsHeader + round256(o) + 2 * round256(l);
}

// ---- TMA tensor maps --------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// A bf16 [B, L, H, D] tensor viewed as 5-D so that one box is `box_rows` consecutive
// local rows of one shard and 64 features of one head (128-byte swizzled rows):
//   striped    dims (D, H, P, n, B):  token = local * P + shard
//   contiguous dims (D, H, n, P, B):  token = shard * n + local
//   zigzag     dims (D, H, c, 2P, B): token = chunk * c + row, c = n / 2 (the kernels
//              pick chunk = shard or 2P-1-shard from the local row)
// (strides increase with the dimension index in every view).
// `heads` is the tensor's own head count (H for q, out, dout; H_kv for k, v).
ra_status_t make_rows_map(CUtensorMap* m, const void* base, const ra_params_t* p, int heads,
                          int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return fail(RA_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t D = p->head_dim, H = heads, P = p->P, B = p->batch;
  const cuuint64_t L = p->seq_len, n = L / P;
  cuuint64_t dims[5], strides[4];
  cuuint32_t box[5], es[5] = {1, 1, 1, 1, 1};
  dims[0] = D;
  dims[1] = H;
  dims[4] = B;
  strides[0] = D * 2;
  strides[3] = L * H * D * 2;
  box[0] = 64;
  box[1] = 1;
  box[4] = 1;
  if (p->layout == RA_LAYOUT_STRIPED) {
    dims[2] = P;
    dims[3] = n;
    strides[1] = H * D * 2;
    strides[2] = P * H * D * 2;
    box[2] = 1;
    box[3] = box_rows;
  } else {
    const cuuint64_t rows = (p->layout == RA_LAYOUT_ZIGZAG) ? n / 2 : n;
    dims[2] = rows;
    dims[3] = L / rows;
    strides[1] = H * D * 2;
    strides[2] = rows * H * D * 2;
    box[2] = box_rows;
    box[3] = 1;
  }
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(RA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return RA_OK;
}

// ---- host work model (closed forms over the whole ring schedule) -----------------
void work_model(const ra_params_t* p, unsigned long long* outp) {
  const int P = p->P, blk = p->block;
  const long long L = p->seq_len, n = L / P;
  const long long Tb = n / blk;
  unsigned long long* tiles = outp;
  unsigned long long* pairs = outp + P;
  unsigned long long* visits = outp + 2 * P;
  for (int i = 0; i < P; ++i) {
    unsigned long long t = 0, pr = 0, v = 0;
    const unsigned long long R = (unsigned long long)n;
    const unsigned long long sum_a = R * (R - 1) / 2;
    for (int k = 0; k < P; ++k) {
      const int j = ((i - k) % P + P) % P;
      if (!p->causal) {
        t += (unsigned long long)(Tb * Tb);
        pr += R * n;
      } else if (p->layout == RA_LAYOUT_STRIPED) {
        // query block tb sees KV blocks u < tb and its diagonal u = tb; with one-token
        // blocks the diagonal's only pair is masked when the KV shard comes later (j > i)
        t += (unsigned long long)(Tb * (Tb + 1) / 2) - ((blk == 1 && j > i) ? (unsigned long long)Tb : 0ull);
        pr += (j <= i) ? sum_a + R : sum_a;
      } else {
        for (long long tb = 0; tb < Tb; ++tb)
          t += blocks_upto(p->layout, j, block_pos(p->layout, i, tb, Tb, P), Tb, P);
        if (p->layout == RA_LAYOUT_CONTIGUOUS)
          pr += (j < i) ? R * n : (j == i ? sum_a + R : 0ull);
        else
          for (long long r = 0; r < n; ++r)
            pr += tokens_upto(p->layout, j, token_of(p->layout, i, r, n, P), n, P);
      }
    }
    for (long long r = 0; r < n; ++r) {
      const long long tok = token_of(p->layout, i, r, n, P);
      v += p->causal ? (unsigned long long)(tok / blk + 1) : (unsigned long long)(L / blk);
    }
    tiles[i] = t;
    pairs[i] = pr;
    visits[i] = v;
  }
}

}  // namespace

void set_last_error_message(const char* msg) { snprintf(g_msg, sizeof(g_msg), "%s", msg); }

ra_status_t encode_2d_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
                           uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return fail(RA_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(RA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return RA_OK;
}

}  // namespace ra

using namespace ra;

extern "C" {

const char* ra_status_string(ra_status_t s) {
  switch (s) {
    case RA_OK: return "RA_OK";
    case RA_ERR_INVALID_ARG: return "RA_ERR_INVALID_ARG";
    case RA_ERR_UNSUPPORTED: return "RA_ERR_UNSUPPORTED";
    case RA_ERR_WORKSPACE: return "RA_ERR_WORKSPACE";
    case RA_ERR_CUDA: return "RA_ERR_CUDA";
    case RA_ERR_DEVICE_TIMEOUT: return "RA_ERR_DEVICE_TIMEOUT";
    case RA_ERR_CHECK: return "RA_ERR_CHECK";
  }
  return "RA_ERR_UNKNOWN";
}

const char* ra_last_error_message(void) { return g_msg; }

size_t ra_fwd_workspace_bytes(const ra_params_t* p) {
  if (check_params(p, true) != RA_OK) return 0;
  return fwd_ws(p);
}

size_t ra_bwd_workspace_bytes(const ra_params_t* p) {
  if (check_params(p, true) != RA_OK) return 0;
  return bwd_ws(p);
}

ra_status_t ra_shard_work_model(const ra_params_t* p, unsigned long long* host_out) {
  ra_status_t s = check_params(p, false);
  if (s != RA_OK) return s;
  if (!host_out) return fail(RA_ERR_INVALID_ARG, "host_out is NULL");
  work_model(p, host_out);
  return RA_OK;
}

ra_status_t ra_fwd(const ra_params_t* p, const void* q, const void* k, const void* v, void* out,
                   int out_dtype, float* lse, unsigned long long* shard_work, void* workspace,
                   size_t workspace_bytes, void* stream) {
  ra_status_t s = check_params(p, true);
  if (s != RA_OK) return s;
  if (!q || !k || !v || !out || !lse) return fail(RA_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
    return fail(RA_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (shard_work && (reinterpret_cast<uintptr_t>(shard_work) & 7u))
    return fail(RA_ERR_INVALID_ARG, "shard_work must be 8-byte aligned");
  if (out_dtype != RA_BF16 && out_dtype != RA_FP32)
    return fail(RA_ERR_INVALID_ARG, "out_dtype must be RA_BF16 or RA_FP32");
  const size_t need = fwd_ws(p);
  if (!workspace || workspace_bytes < need || !aligned16(workspace))
    return fail(RA_ERR_WORKSPACE, "workspace needs %zu bytes (16-byte aligned), got %zu", need,
                workspace_bytes);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  CUtensorMap tq, tk, tv;
  if ((s = make_rows_map(&tq, q, p, p->heads, kTile)) != RA_OK) return s;
  if ((s = make_rows_map(&tk, k, p, kv_of(p), kTile)) != RA_OK) return s;
  if ((s = make_rows_map(&tv, v, p, kv_of(p), kTile)) != RA_OK) return s;

  FwdArgs a{};
  a.B = p->batch;
  a.H = p->heads;
  a.G = p->heads / kv_of(p);
  a.D = p->head_dim;
  a.P = p->P;
  a.layout = p->layout;
  a.causal = p->causal;
  a.block = p->block;
  a.L = p->seq_len;
  a.n = (int)(p->seq_len / p->P);
  a.T = a.n / kTile;
  a.npair = npair_of(p);
  a.n_split = n_split_of(p);
  a.scale_log2 = scale_of(p) * 1.4426950408889634f;
  a.out = out;
  a.out_fp32 = out_dtype == RA_FP32;
  a.lse = lse;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.err = reinterpret_cast<unsigned int*>(ws);
  if (a.n_split > 1) {
    const size_t o = (size_t)p->batch * p->seq_len * p->heads * p->head_dim * 4;
    a.o_part = reinterpret_cast<float*>(ws + kWsHeader);
    a.lse_part = reinterpret_cast<float*>(ws + kWsHeader + round256(a.n_split * o));
  }
  a.shard_work = shard_work;
  a.wait_limit_ns = kWaitLimitNs;
  cudaError_t e;
  if (shard_work) {
    e = cudaMemsetAsync(shard_work, 0, sizeof(unsigned long long) * 3 * p->P, st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(shard_work)");
  }
  e = launch_fwd(a, tq, tk, tv, st);
  if (e != cudaSuccess) return cuda_fail(e, "forward kernel launch");
  if (a.n_split > 1) {
    e = launch_merge(a.n_split, a.o_part, a.lse_part, a.B, a.L, a.H, a.D, out, a.out_fp32, lse, st);
    if (e != cudaSuccess) return cuda_fail(e, "merge kernel launch");
  }
  return RA_OK;
}

}  // extern "C"

namespace ra {
namespace {

// Workspace layout of the backward: [header | dQ fp32 [B,L,H,D] | D [B,H,P,n] | lse2].
struct BwdWs {
  float* dq_acc;
  float* Dsm;
  float* L2sm;
  size_t o, l;
};

ra_status_t bwd_common(const ra_params_t* p, void* workspace, size_t workspace_bytes,
                       BwdWs* w) {
  ra_status_t s = check_params(p, true);
  if (s != RA_OK) return s;
  const size_t need = bwd_ws(p);
  if (!workspace || workspace_bytes < need || !aligned16(workspace))
    return fail(RA_ERR_WORKSPACE, "workspace needs %zu bytes (16-byte aligned), got %zu", need,
                workspace_bytes);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  w->o = (size_t)p->batch * p->seq_len * p->heads * p->head_dim;
  w->l = (size_t)p->batch * p->heads * p->seq_len;
  w->dq_acc = reinterpret_cast<float*>(ws + kWsHeader);
  w->Dsm = reinterpret_cast<float*>(ws + kWsHeader + round256(w->o * 4));
  w->L2sm = reinterpret_cast<float*>(ws + kWsHeader + round256(w->o * 4) + round256(w->l * 4));
  return RA_OK;
}

}  // namespace
}  // namespace ra

extern "C" {

ra_status_t ra_bwd_preprocess(const ra_params_t* p, const void* out, int out_dtype,
                              const float* lse, const void* dout, void* workspace,
                              size_t workspace_bytes, void* stream) {
  BwdWs w;
  ra_status_t s = bwd_common(p, workspace, workspace_bytes, &w);
  if (s != RA_OK) return s;
  if (!out || !lse || !dout) return fail(RA_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned16(out) || !aligned16(lse) || !aligned16(dout))
    return fail(RA_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (out_dtype != RA_BF16 && out_dtype != RA_FP32)
    return fail(RA_ERR_INVALID_ARG, "out_dtype must be RA_BF16 or RA_FP32");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // one kernel: D, lse * log2(e) (shard-major, negated) and the zeroed dQ accumulator
  cudaError_t e = launch_bwd_pre(out, out_dtype == RA_FP32, dout, lse, w.Dsm, w.L2sm, w.dq_acc,
                                 p->batch, p->seq_len, p->heads, p->head_dim, p->P, p->layout,
                                 st);
  if (e != cudaSuccess) return cuda_fail(e, "backward preprocess launch");
  return RA_OK;
}

ra_status_t ra_bwd_main(const ra_params_t* p, const void* q, const void* k, const void* v,
                        const void* dout, void* dk, void* dv, void* workspace,
                        size_t workspace_bytes, void* stream) {
  BwdWs w;
  ra_status_t s = bwd_common(p, workspace, workspace_bytes, &w);
  if (s != RA_OK) return s;
  if (!q || !k || !v || !dout || !dk || !dv) return fail(RA_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dout) || !aligned16(dk) ||
      !aligned16(dv))
    return fail(RA_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  CUtensorMap tq, tk, tv, tdo;
  if ((s = make_rows_map(&tq, q, p, p->heads, kTile)) != RA_OK) return s;
  if ((s = make_rows_map(&tk, k, p, kv_of(p), kTile)) != RA_OK) return s;
  if ((s = make_rows_map(&tv, v, p, kv_of(p), kTile)) != RA_OK) return s;
  if ((s = make_rows_map(&tdo, dout, p, p->heads, kTile)) != RA_OK) return s;
  BwdArgs a{};
  a.B = p->batch;
  a.H = p->heads;
  a.Hkv = kv_of(p);
  a.G = p->heads / a.Hkv;
  a.D = p->head_dim;
  a.P = p->P;
  a.layout = p->layout;
  a.causal = p->causal;
  a.L = p->seq_len;
  a.n = (int)(p->seq_len / p->P);
  a.T = a.n / kTile;
  a.scale = scale_of(p);
  a.scale_log2 = a.scale * 1.4426950408889634f;
  a.lse = w.L2sm;
  a.Dvec = w.Dsm;
  a.dq_acc = w.dq_acc;
  a.dk = dk;
  a.dv = dv;
  a.err = static_cast<unsigned int*>(workspace);
  a.wait_limit_ns = kWaitLimitNs;
  cudaError_t e = launch_bwd(a, tq, tk, tv, tdo, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "backward kernel launch");
  return RA_OK;
}

ra_status_t ra_bwd_finalize(const ra_params_t* p, void* dq, void* workspace,
                            size_t workspace_bytes, void* stream) {
  BwdWs w;
  ra_status_t s = bwd_common(p, workspace, workspace_bytes, &w);
  if (s != RA_OK) return s;
  if (!dq || !aligned16(dq)) return fail(RA_ERR_INVALID_ARG, "dq must be a 16-byte aligned pointer");
  cudaError_t e = launch_dq_convert(w.dq_acc, dq, scale_of(p), w.o,
                                    reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "dq convert launch");
  return RA_OK;
}

ra_status_t ra_bwd(const ra_params_t* p, const void* q, const void* k, const void* v,
                   const void* out, int out_dtype, const float* lse, const void* dout, void* dq,
                   void* dk, void* dv, void* workspace, size_t workspace_bytes, void* stream) {
  // validate everything before the first launch
  BwdWs w;
  ra_status_t s = bwd_common(p, workspace, workspace_bytes, &w);
  if (s != RA_OK) return s;
  if (!q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv)
    return fail(RA_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse) ||
      !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return fail(RA_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (out_dtype != RA_BF16 && out_dtype != RA_FP32)
    return fail(RA_ERR_INVALID_ARG, "out_dtype must be RA_BF16 or RA_FP32");
  s = ra_bwd_preprocess(p, out, out_dtype, lse, dout, workspace, workspace_bytes, stream);
  if (s != RA_OK) return s;
  s = ra_bwd_main(p, q, k, v, dout, dk, dv, workspace, workspace_bytes, stream);
  if (s != RA_OK) return s;
  return ra_bwd_finalize(p, dq, workspace, workspace_bytes, stream);
}

ra_status_t ra_merge(int n_parts, const float* o_parts, const float* lse_parts, int batch,
                     int64_t seq_len, int heads, int head_dim, void* out, int out_dtype,
                     float* lse, void* stream) {
  if (n_parts < 1 || batch < 1 || seq_len < 1 || heads < 1)
    return fail(RA_ERR_INVALID_ARG, "n_parts, batch, seq_len, heads must be >= 1");
  if (head_dim < 8 || head_dim > 256 || head_dim % 8 != 0)
    return fail(RA_ERR_INVALID_ARG, "head_dim must be a multiple of 8 in [8, 256]");
  if (!o_parts || !lse_parts || !out || !lse) return fail(RA_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(o_parts) || !aligned16(out)) return fail(RA_ERR_INVALID_ARG, "misaligned pointer");
  if (out_dtype != RA_BF16 && out_dtype != RA_FP32)
    return fail(RA_ERR_INVALID_ARG, "out_dtype must be RA_BF16 or RA_FP32");
  cudaError_t e = launch_merge(n_parts, o_parts, lse_parts, batch, seq_len, heads, head_dim, out,
                               out_dtype == RA_FP32, lse, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "merge kernel launch");
  return RA_OK;
}

ra_status_t ra_check_error(void* workspace, void* stream) {
  if (!workspace) return fail(RA_ERR_INVALID_ARG, "workspace is NULL");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned int word = 0;
  e = cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "reading the workspace error word");
  if (word != 0) {
    e = cudaMemset(workspace, 0, sizeof(word));
    if (e != cudaSuccess) return cuda_fail(e, "clearing the workspace error word");
    if (word & 0x10u)
      return fail(RA_ERR_CUDA, "the backward kernel found its shared-memory base not 1024-byte "
                  "aligned and did nothing (error word 0x%x)", word);
    if (word & kChkMask)
      return fail(RA_ERR_CHECK, "a range check of the checked build failed (error word 0x%x: "
                  "0x100 TMA box, 0x200 TMEM, 0x400 shared memory, 0x800 global index, "
                  "0x1000 item count)", word);
    return fail(RA_ERR_DEVICE_TIMEOUT, "a kernel gave up a bounded wait (error word 0x%x)", word);
  }
  return RA_OK;
}

ra_status_t ra_selftest_timeout(void* workspace, size_t workspace_bytes, unsigned int timeout_us,
                                void* stream) {
  if (!workspace || workspace_bytes < kWsHeader || !aligned16(workspace))
    return fail(RA_ERR_WORKSPACE, "workspace needs %zu bytes", (size_t)kWsHeader);
  if (timeout_us == 0 || timeout_us > 10000000u)
    return fail(RA_ERR_INVALID_ARG, "timeout_us must be in [1, 10^7]");
  cudaError_t e = launch_selftest_timeout(static_cast<unsigned int*>(workspace),
                                          (uint64_t)timeout_us * 1000ull,
                                          reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "self-test kernel launch");
  return RA_OK;
}

int ra_checks_enabled(void) { return kChecked ? 1 : 0; }

ra_status_t ra_selftest_exp2(const float* x, float* y_soft, float* y_hw, long long n,
                             void* stream) {
  if (!x || !y_soft || !y_hw) return fail(RA_ERR_INVALID_ARG, "null pointer");
  if (n < 1 || n >= (1LL << 31)) return fail(RA_ERR_INVALID_ARG, "n must be in [1, 2^31)");
  cudaError_t e =
      launch_selftest_exp2(x, y_soft, y_hw, n, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "self-test kernel launch");
  return RA_OK;
}

}  // extern "C"
