/*
 * ra.h -- C ABI of libra: exact blockwise ring attention (contiguous, striped and
 * zigzag layouts) over P virtual shards held on one GPU, for NVIDIA GB300 (sm_103a).
 *
 * The method (sources are four web pages on Ring Attention / Striped Attention):
 *   - "Ring Attention 論文分析" (labhub): blockwise attention with an online softmax
 *     (section "ブロック単位の分割戦略"), the ring forward (section "リングトポロジーと
 *     KV の循環"), causal block skipping (section "Causal Masking の処理"), the
 *     backward with recomputed scores (sections "逆伝播での KV 再循環" and
 *     "チェックポインティング戦略").
 *   - "Ring Attention: Sequence Parallelism for Long Context" (vanos001): ring order
 *     (step k: shard i attends KV shard (i - k) mod P), the striped assignment
 *     (token r -> shard r mod P, section "The Causal-Mask Problem: Striped
 *     Attention"), the zigzag assignment (same section: two half-shards placed
 *     symmetrically near the start and the end of the sequence), and the per-device
 *     work count of section "Worked Demo".
 *
 * One call covers all P shards: the pages' per-device ring becomes a schedule inside
 * one kernel, and a "hop" is a tile load of KV shard (i - k) mod P from device memory.
 *
 * Conventions for every entry point:
 *   - Tensors are row-major.  q, out, dout, dq are [B, L, H, D] and k, v, dk, dv are
 *     [B, L, H_kv, D] (H_kv = H unless kv_heads says otherwise), with
 *     tokens in NATURAL order for every layout (the shard permutation is internal;
 *     attention is permutation-equivariant, aibr.jp Striped Attention summary, §3).
 *     lse is float32 [B, H, L], natural logarithm.
 *   - All pointers are DEVICE pointers unless stated otherwise, 16-byte aligned.
 *     The caller owns all memory; the library keeps no allocation between calls.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Compute calls are asynchronous on it.
 *   - Argument errors are detected on the host, before any launch, and returned as
 *     RA_ERR_INVALID_ARG / RA_ERR_UNSUPPORTED / RA_ERR_WORKSPACE; nothing is written.
 *     A failed CUDA runtime call returns RA_ERR_CUDA.  Device-side timeouts (every
 *     wait in the kernels is bounded) are recorded in the workspace's error word and
 *     reported by ra_check_error().  No exception or abort crosses this ABI.
 *   - ra_last_error_message() returns a thread-local text for the last failure.
 */
#ifndef RA_H_
#define RA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  RA_OK = 0,
  RA_ERR_INVALID_ARG = 1,     /* null/misaligned pointer, bad size or enum value  */
  RA_ERR_UNSUPPORTED = 2,     /* valid request this build has no kernel for       */
  RA_ERR_WORKSPACE = 3,       /* workspace null or smaller than *_workspace_bytes */
  RA_ERR_CUDA = 4,            /* a CUDA runtime/driver call failed                */
  RA_ERR_DEVICE_TIMEOUT = 5,  /* a bounded wait inside a kernel ran out           */
  RA_ERR_CHECK = 6            /* checked build: a kernel found an index out of range */
} ra_status_t;

typedef enum {
  RA_LAYOUT_CONTIGUOUS = 0,
  RA_LAYOUT_STRIPED = 1,
  RA_LAYOUT_ZIGZAG = 2
} ra_layout_t;
typedef enum { RA_BF16 = 0, RA_FP32 = 1 } ra_dtype_t;

/*
 * Problem description.
 *   batch, heads     B, H >= 1.
 *   seq_len          L >= 1, divisible by P * block (the pages assume equal shards,
 *                    labhub section "長文データの前処理とチャンク割り当て"; there is
 *                    no padding here); ZIGZAG needs L divisible by 2 * P * block.
 *   head_dim         D in {64, 128}.
 *   block            the blockwise loop's block size (BPT block_size), {128, 256}.
 *                    The result does not depend on it beyond rounding order; it sets
 *                    the unit of the work counter's "tiles".
 *   P                number of virtual shards (ring length), 1 <= P <= 1024.
 *   layout           ra_layout_t: CONTIGUOUS (token t -> shard t / (L/P)),
 *                    STRIPED (token t -> shard t mod P) or ZIGZAG (the sequence cut
 *                    into 2P chunks of c = L/(2P) tokens; shard i holds chunks i and
 *                    2P-1-i, local rows [0, c) and [c, 2c) in that order).
 *   causal           0 or 1 (key c visible to query r iff c <= r, original positions).
 *   softmax_scale    > 0, or 0 for 1/sqrt(D).
 *   n_split          forward only: 1 = one online-softmax state carried over all P
 *                    ring steps; g > 1 (g divides P) = the ring steps are cut into g
 *                    groups, each writing a partial (O_g, lse_g) that ra_merge then
 *                    combines; 0 = let the library choose.
 *   kv_heads         H_kv, the number of key/value heads: 0 (or H) for plain multi-head
 *                    attention, otherwise a divisor of H (grouped-query attention; 1 is
 *                    MQA).  Query head h attends with key/value head h / (H / H_kv), i.e.
 *                    G = H / H_kv consecutive query heads share one; the gradient of a
 *                    shared head is the sum over its G query heads (labhub, comparison
 *                    section "比較分析": ring attention is fully compatible with GQA/MQA).
 * Size limits: B * L * H * D <= 2^40 elements and B * H * L <= 2^36 rows.  A violated
 * rule is RA_ERR_INVALID_ARG, except a head_dim or block outside the sets above
 * (RA_ERR_UNSUPPORTED: a valid request with no kernel).
 */
typedef struct {
  int batch;
  int64_t seq_len;
  int heads;
  int head_dim;
  int block;
  int P;
  int layout;
  int causal;
  float softmax_scale;
  int n_split;
  int kv_heads;
} ra_params_t;

/* Bytes of device workspace ra_fwd / ra_bwd need for `p` (0 if `p` is invalid).
 * The workspace must be zero-filled before its first use; afterwards the library
 * keeps its error word consistent (ra_check_error re-zeroes it). */
size_t ra_fwd_workspace_bytes(const ra_params_t* p);
size_t ra_bwd_workspace_bytes(const ra_params_t* p);

/*
 * Forward: out = softmax(scale * q k^T, causal mask) v, lse = log-sum-exp of the
 * scaled, masked scores, computed ring-wise: the queries of shard i visit KV shards
 * (i - k) mod P for k = 0..P-1, KV tiles in order inside a shard, merging with an
 * online softmax (labhub, sections "ブロック単位の分割戦略" and "リングトポロジーと KV
 * の循環"); causal KV tiles entirely after the query tile are skipped, the diagonal
 * ones masked (labhub, section "Causal Masking の処理").
 *   q, k, v      bf16 [B, L, H, D].
 *   out          [B, L, H, D] of out_dtype (bf16: round to nearest even).
 *   lse          fp32 [B, H, L]; -inf for a row with no visible key.
 *   shard_work   NULL, or device uint64 [3][P] overwritten with the per-shard work the
 *                kernel executed: [0][i] (Q block, KV block) pairs of `block` tokens
 *                computed for the queries of shard i (causal: those holding at least
 *                one visible (query, key) pair; all otherwise), [1][i] unmasked (query, key)
 *                pairs, [2][i] the vanos001 "Worked Demo" unit (per query row, KV
 *                blocks in natural order holding a visible key).
 *   workspace    device buffer of >= ra_fwd_workspace_bytes(p) bytes.
 */
ra_status_t ra_fwd(const ra_params_t* p, const void* q, const void* k, const void* v,
                   void* out, int out_dtype, float* lse,
                   unsigned long long* shard_work,
                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward (labhub, section "逆伝播での KV 再循環"): with D_r = dO_r . O_r,
 * P = exp(scale q k^T - lse) (0 where masked), dV = P^T dO, dP = dO V^T,
 * dS = P * (dP - D) * scale, dQ = dS K, dK = dS^T Q.  Scores are recomputed from
 * q, k and lse (section "チェックポインティング戦略"); each KV tile stays resident
 * while the query tiles pass it in ring order (the pages' "dK, dV back to the owner"
 * becomes on-chip accumulation).
 *   q, k, v, dout  bf16 [B, L, H, D];  out [B, L, H, D] of out_dtype;  lse from ra_fwd.
 *   dq, dk, dv     bf16 [B, L, H, D] outputs (fp32 accumulation inside).
 *   workspace      device buffer of >= ra_bwd_workspace_bytes(p) bytes (holds the
 *                  fp32 dQ accumulator and D).
 */
ra_status_t ra_bwd(const ra_params_t* p, const void* q, const void* k, const void* v,
                   const void* out, int out_dtype, const float* lse, const void* dout,
                   void* dq, void* dk, void* dv,
                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * The three stages ra_bwd runs, callable one by one (same kernels, same workspace):
 *   ra_bwd_preprocess  D = rowsum(dO * O) and lse * log2(e), both stored negated and shard-major
 *                      ([B, H, P, L/P] fp32) in the workspace; zeroes the fp32 dQ
 *                      accumulator (labhub, "逆伝播での KV 再循環": the D vector).
 *   ra_bwd_main        the ring backward proper: writes dk, dv (bf16) and accumulates
 *                      unscaled dQ into the workspace.  Needs the preprocess results.
 *   ra_bwd_finalize    dq = bf16(scale * accumulated dQ).
 * Arguments have the meaning given for ra_bwd; the same workspace must be passed to all
 * three, in this order, on one stream.
 */
ra_status_t ra_bwd_preprocess(const ra_params_t* p, const void* out, int out_dtype,
                              const float* lse, const void* dout, void* workspace,
                              size_t workspace_bytes, void* stream);
ra_status_t ra_bwd_main(const ra_params_t* p, const void* q, const void* k, const void* v,
                        const void* dout, void* dk, void* dv, void* workspace,
                        size_t workspace_bytes, void* stream);
ra_status_t ra_bwd_finalize(const ra_params_t* p, void* dq, void* workspace,
                            size_t workspace_bytes, void* stream);

/*
 * Merge of normalised partials (the online-softmax correction of labhub section
 * "ブロック単位の分割戦略", applied to whole partial results):
 *   lse = ln sum_g exp(lse_g),  out = sum_g exp(lse_g - lse) O_g,
 * skipping partials with lse_g = -inf; a row whose partials are all -inf gets
 * out = 0, lse = -inf.
 *   o_parts    fp32 [n_parts][B, L, H, D];  lse_parts fp32 [n_parts][B, H, L].
 *   out        [B, L, H, D] of out_dtype;   lse fp32 [B, H, L].
 * head_dim must be a multiple of 8 and <= 256.
 */
ra_status_t ra_merge(int n_parts, const float* o_parts, const float* lse_parts,
                     int batch, int64_t seq_len, int heads, int head_dim,
                     void* out, int out_dtype, float* lse, void* stream);

/*
 * Closed-form per-shard work for `p` in the units of ra_fwd's shard_work, written to
 * HOST memory host_out[3 * P].  Any block >= 1 dividing L / P is accepted here (the
 * GPU path needs {128, 256}); with L = 32, P = 4, block = 8, causal, unit [2] gives
 * the vanos001 demo's 8/16/24/32 (contiguous) and 20/20/20/20 (striped).
 */
ra_status_t ra_shard_work_model(const ra_params_t* p, unsigned long long* host_out);

/*
 * Backward without a workspace, for callers that cannot allocate device memory: a
 * plugin whose host runtime hands it tensors and a stream but no allocator, or a
 * latency-critical caller that may not call cudaMalloc on its hot path (the call can
 * synchronise the device and its cost is unbounded).  The pages have no counterpart of
 * this entry point; it is a deployment convenience.
 *   Same computation and arguments as ra_bwd, minus the workspace: the scratch (error
 *   word, fp32 dQ accumulator, D, lse * log2(e)) lives in one 64 MiB array of device
 *   memory inside the library, which every GPU that loads the library holds until the
 *   process exits.  Problems whose ra_bwd_workspace_bytes() exceeds 64 MiB are rejected
 *   with RA_ERR_WORKSPACE (roughly B * L * H above 128K rows at head_dim 128, 256K at 64).
 *   The first call on a device looks up the array's device address with that device
 *   current (set-up); make that first call before any stream capture.
 *   Nothing is allocated: no cudaMalloc, cudaFree or allocating library call.
 *   All calls share the one array, and it keeps the last call's contents: each call
 *   clears the error word and zeroes the dQ accumulator itself.  Calls that overlap on
 *   the GPU (two streams, or two threads) race on the array and corrupt each other;
 *   serialise them.  A device-side timeout of one call is cleared by the next call, so
 *   it is not reported through this entry point (use ra_bwd + ra_check_error for that).
 */
ra_status_t ra_bwd_noalloc(const ra_params_t* p, const void* q, const void* k, const void* v,
                           const void* out, int out_dtype, const float* lse, const void* dout,
                           void* dq, void* dk, void* dv, void* stream);

/* Synchronises `stream`, reads the workspace's device error word, re-zeroes it, and
 * returns RA_ERR_DEVICE_TIMEOUT if a kernel gave up a wait since the last check, and
 * RA_ERR_CHECK if (checked build only) a kernel found an index out of range. */
ra_status_t ra_check_error(void* workspace, void* stream);

/* Diagnostic for the bounded-wait machinery: launches one CTA that waits on a
 * barrier nothing arrives on, with a `timeout_us` limit; the kernel records the
 * timeout in the workspace error word and returns normally (no trap, the context
 * stays usable).  ra_check_error() then returns RA_ERR_DEVICE_TIMEOUT. */
ra_status_t ra_selftest_timeout(void* workspace, size_t workspace_bytes,
                                unsigned int timeout_us, void* stream);

/* Self-test of the two 2^x forms the softmax kernels mix (no counterpart on the pages,
 * which take exp as given): for each of n fp32 inputs x[i] (device memory),
 * y_soft[i] = the software form (range reduction and a polynomial on the FMA pipe,
 * relative error below 4e-6; x <= -127 gives +0, NaN gives NaN) and y_hw[i] = the
 * hardware unit's ex2.approx.ftz.  x, y_soft, y_hw: device fp32 arrays of n elements,
 * caller-owned, 4-byte aligned; n in [1, 2^31).  Asynchronous on `stream`.  Returns
 * RA_ERR_INVALID_ARG for null pointers or n out of range, RA_ERR_CUDA if the launch fails. */
ra_status_t ra_selftest_exp2(const float* x, float* y_soft, float* y_hw, long long n,
                             void* stream);

/* 1 if this library is the checked build (compiled with RA_CHECKS, e.g. libra_checked.so),
 * 0 otherwise.  In the checked build every kernel tests its tile and TMA box coordinates,
 * TMEM columns and lane quarters, shared-memory operand offsets, global element indices
 * and the per-role item counts before use; a violation skips the access, sets a bit of the
 * workspace error word and ra_check_error() returns RA_ERR_CHECK.  It stands in for a
 * memory checker; the pages have no counterpart. */
int ra_checks_enabled(void);

const char* ra_status_string(ra_status_t s);
const char* ra_last_error_message(void);

/* ==================================================================================
 * Blockwise Parallel Transformer layer, forward (labhub, section "BPT の Feedforward
 * 融合"): Q, K, V projections, the ring attention above, then per block of rows the
 * output projection, residual + LayerNorm, the feed-forward network (Linear, GELU,
 * Linear), residual + LayerNorm:
 *   h1  = LN1(x + attention(x Wq^T + bq, x Wk^T + bk, x Wv^T + bv) Wo^T + bo)
 *   out = LN2(h1 + GELU(h1 W1^T + b1) W2^T + b2)
 * Post-norm as on the page; LN uses the biased variance; GELU is the exact erf form.
 * Only one block's feed-forward intermediates exist at a time, so the workspace grows
 * with block_rows * d_ff, not with seq_len * d_ff.
 * ================================================================================== */

typedef enum {
  RA_EPI_BIAS = 0,           /* out bf16 = x W^T + b                        */
  RA_EPI_BIAS_GELU = 1,      /* out bf16 = GELU(x W^T + b)                  */
  RA_EPI_BIAS_RESIDUAL = 2   /* out fp32 = x W^T + b + residual (bf16 [rows, out]) */
} ra_epilogue_t;

/*
 * A Linear layer on tcgen05 tensor cores with its elementwise epilogue fused:
 *   x [rows, in_features] bf16, weight [out_features, in_features] bf16 (torch.nn.Linear
 *   layout), bias [out_features] fp32, residual (RA_EPI_BIAS_RESIDUAL only) [rows,
 *   out_features] bf16, out [rows, out_features] bf16 or fp32 as listed above.
 *   rows % 128 == 0, out_features % 256 == 0, in_features % 64 == 0 (else
 *   RA_ERR_UNSUPPORTED); device pointers, 16-byte aligned.  workspace: >= 256 bytes,
 *   zero-filled before first use; its first word is the error word (ra_check_error).
 */
ra_status_t ra_linear(int64_t rows, int in_features, int out_features, const void* x,
                      const void* weight, const float* bias, const void* residual, int epilogue,
                      void* out, void* workspace, size_t workspace_bytes, void* stream);

/*
 * LayerNorm over the last dimension: out = (x - mean) / sqrt(var + eps) * gamma + beta,
 * var the biased variance.  x fp32 [rows, features]; gamma, beta fp32 [features]; out
 * [rows, features] of out_dtype.  features % 512 == 0 and <= 8192 (else
 * RA_ERR_UNSUPPORTED); eps > 0.
 */
ra_status_t ra_layernorm(int64_t rows, int features, const float* x, const float* gamma,
                         const float* beta, float eps, void* out, int out_dtype, void* stream);

/*
 * Layer description.
 *   attn        the attention: batch, seq_len, heads, head_dim (d_model = heads *
 *               head_dim), block, P, layout, causal, softmax_scale, n_split, kv_heads as
 *               for ra_fwd.  With kv_heads = H_kv < heads the K and V projections are
 *               H_kv * head_dim wide (grouped-query attention); H_kv * head_dim must be a
 *               multiple of 256.
 *   d_ff        feed-forward width, a positive multiple of 256.
 *   block_rows  rows of the flattened [batch * seq_len] sequence per post-attention
 *               block, a multiple of 128; 0 = min(batch * seq_len, 16384).
 *   ln_eps      LayerNorm epsilon (>= 0), 0 = 1e-5.
 * d_model must be a multiple of 512 and at most 8192.
 */
typedef struct {
  ra_params_t attn;
  int d_ff;
  int64_t block_rows;
  float ln_eps;
} ra_bpt_params_t;

/* Layer parameters, all device pointers: weights bf16 in torch.nn.Linear layout
 * [out, in] (wq, wo [d, d]; wk, wv [H_kv * head_dim, d]; w1 [d_ff, d]; w2 [d, d_ff]),
 * biases and LayerNorm scales / shifts fp32. */
typedef struct {
  const void* wq;
  const void* wk;
  const void* wv;
  const void* wo;
  const void* w1;
  const void* w2;
  const float* bq;
  const float* bk;
  const float* bv;
  const float* bo;
  const float* b1;
  const float* b2;
  const float* ln1_g;
  const float* ln1_b;
  const float* ln2_g;
  const float* ln2_b;
} ra_bpt_weights_t;

/* Bytes of workspace ra_bpt_fwd needs (0 if `p` is invalid): the attention's workspace
 * (sized for its forward and backward; its error word is the layer's), Q, K, V and the
 * attention output (bf16 [B*L, d] each), lse, and one block's fp32 [block_rows, d] and
 * bf16 [block_rows, d] and [block_rows, d_ff] buffers.  Zero-filled before first use. */
size_t ra_bpt_workspace_bytes(const ra_bpt_params_t* p);

/* x [batch, seq_len, d] bf16 (tokens in natural order), out same shape of out_dtype. */
ra_status_t ra_bpt_fwd(const ra_bpt_params_t* p, const void* x, const ra_bpt_weights_t* w,
                       void* out, int out_dtype, void* workspace, size_t workspace_bytes,
                       void* stream);

/* Gradients of the layer, all device pointers: dx bf16 [batch, seq_len, d]; the others
 * fp32, shaped like the parameter of the same name.  ra_bpt_bwd overwrites every one. */
typedef struct {
  void* dx;
  float* wq;
  float* wk;
  float* wv;
  float* wo;
  float* w1;
  float* w2;
  float* bq;
  float* bk;
  float* bv;
  float* bo;
  float* b1;
  float* b2;
  float* ln1_g;
  float* ln1_b;
  float* ln2_g;
  float* ln2_b;
} ra_bpt_grads_t;

/* Bytes of workspace for a forward followed by a backward (>= ra_bpt_workspace_bytes; the
 * forward's part of the layout is the same), 0 if `p` is invalid or has no backward
 * kernel (d_model must be at most 4096). */
size_t ra_bpt_train_workspace_bytes(const ra_bpt_params_t* p);

/*
 * Backward of the layer: given dout (bf16 [batch, seq_len, d]) = d loss / d out, writes
 * every gradient of `g`.  Must follow ra_bpt_fwd on the same x, weights and workspace
 * (whose Q, K, V, attention output and lse it reuses); the workspace must hold
 * ra_bpt_train_workspace_bytes.  Per block of rows it recomputes the forward's Wo,
 * LayerNorm, W1 and W2 steps (memory stays per block), then runs the LayerNorm, GELU and
 * Linear backward steps (weight gradients accumulated in fp32 across blocks), and finally
 * the attention backward (ra_bwd) over the whole sequence and the projections' backward.
 */
ra_status_t ra_bpt_bwd(const ra_bpt_params_t* p, const void* x, const ra_bpt_weights_t* w,
                       const void* dout, const ra_bpt_grads_t* g, void* workspace,
                       size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* RA_H_ */
