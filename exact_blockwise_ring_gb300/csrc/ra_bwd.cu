// ra_bwd.cu -- backward kernel of exact blockwise ring attention on tcgen05 tensor cores.
//
// Method (labhub "Ring Attention 論文分析", section "逆伝播での KV 再循環"): with
// D = rowsum(dO * O) and the forward's lse, per (query block, KV block):
//   P = exp(scale q k^T - lse)   (scores recomputed, section "チェックポインティング戦略")
//   dV += P^T dO ;  dP = dO V^T ;  dS = P * (dP - D) * scale ;  dQ += dS K ;  dK += dS^T Q
// The pages send dK/dV partials back to the KV block's owner with a reduce; here the KV
// tile stays resident in one CTA while the query tiles of every shard pass it in ring
// order (shard i = (j + k) mod P at step k for KV shard j), so dK and dV accumulate in
// TMEM and leave once.  dQ partials are added into an fp32 accumulator in global memory.
// For the striped layout at sizes where a head's Q, dO and dQ accumulator exceed half the
// L2, query tiles pass row index by row index instead: for t from the last tile down, the
// shards i = (j + k) mod P in ring order.  The CTAs launched side by side (the same KV tile
// index u of every shard: the same work) then read row t of every shard within P tiles of
// each other, so each query tile and its dQ rows are fetched from DRAM about once per
// group rather than once per CTA (at a million tokens they are several times the L2),
// while at each moment the group's dQ reductions land on different tiles.
//
// One CTA = 128 keys (tile u of shard j) of one (batch, key/value head hk); query tiles of
// 128 rows.  With grouped-query attention the G query heads h = hk*G + g that read this
// key/value head pass one after another (g outermost, then the tile rows and the ring),
// so dK and dV sum over the group in TMEM as they do over the ring.
// Roles (640 threads):
//   warp 0      producer: K, V once (TMA); per query tile Q, dO (TMA) and its 128 lse
//               (log2 domain) and D values (bulk copies from the shard-major arrays the
//               preprocess kernel wrote), two stages
//   warp 1      TMEM allocator and tcgen05.mma issuer (the whole warp walks the issue
//               loop; one elected lane issues)
//   warps 4-11  two warpgroups, thread = key row, warpgroup g takes query columns
//               [64g, 64g+64) in four passes of 16: P^T = exp2(S^T*c - lse2) (bf16, back
//               into TMEM inside its own S^T columns, as the A operand of dV) and
//               dS^T = P^T (dP^T - D) (bf16, 128-byte-swizzled shared tile); at the end
//               warpgroup 0 writes dV, warpgroup 1 writes dK
//   warps 12-19 two warpgroups draining dQ^T (thread = feature row, 64 query columns
//               each) into the fp32 accumulator with coalesced reductions, which then run
//               in the background of the next tiles' work
// MMAs per query tile m (M = 128 TMEM lanes, N = 128):
//   S^T  = K Q^T      A K-major smem,   B K-major smem          -> S region
//   dP^T = V dO^T     A K-major smem,   B K-major smem          -> dP region
//   dV  += P^T dO     A TMEM (P^T),     B MN-major smem (dO)
//   dK  += dS^T Q     A K-major smem,   B MN-major smem (Q)
//   dQ^T = K^T dS^T   A MN-major smem,  B MN-major smem (dS^T)  -> dP region
// Issue order once tile m's scores are consumed: dQ^T(m), dV(m), S^T(m+1), [dQ^T drained],
// dP^T(m+1), dK(m): the drain overlaps dV and S^T, dK(m) overlaps the next tile's scores.
// TMEM columns: S^T/P^T [0,128), dP^T/dQ^T [128,256), dV [256,384), dK [384,512).
#include <cuda_bf16.h>

#include "ra_check.cuh"
#include "ra_internal.h"
#include "ra_ptx.cuh"
#include "ra_rows.cuh"

namespace ra {

namespace {

constexpr int BQ = 128;     // query rows per tile
constexpr int NSTQ = 2;     // query-side pipeline stages

// D_ = head dim (64 or 128).  K stays resident 128 features wide: with D_ = 64 its
// features [64, 128) are zero, so that dQ^T = K^T dS^T keeps M = 128 (rows [64, 128) of
// the product are zero and are not drained).
template <int D_>
struct BwdCfg {
  static constexpr int KB = kTile * 128 * 2;       // K tile bytes in shared memory (32 KB)
  static constexpr int VB = kTile * D_ * 2;        // V tile bytes, also the K bytes loaded
  static constexpr int QB = BQ * D_ * 2;           // Q or dO tile bytes
  static constexpr int SB = kTile * BQ * 2;        // dS^T tile bytes (32 KB)
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KB;
  static constexpr int OFF_Q = OFF_V + VB;
  static constexpr int OFF_DO = OFF_Q + NSTQ * QB;
  static constexpr int OFF_DS = OFF_DO + NSTQ * QB;
  static constexpr int OFF_LD = OFF_DS + SB;       // per stage: 128 lse2 + 128 D floats
  static constexpr int LDB = 2 * BQ * 4;
  static constexpr int OFF_BAR = OFF_LD + NSTQ * LDB;
  // kv_full, q_full[NSTQ], q_empty[NSTQ], s_full, ds_ready, ds_free, dq_full, dq_empty,
  // kv_final, drain
  static constexpr int NBAR = 1 + 2 * NSTQ + 7;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  // no alignment slack: the kernel requires (and checks) a 1024-byte aligned base
  static constexpr int SMEM_BYTES = OFF_MISC + 64;
  static constexpr int COL_S = 0, COL_DP = 128, COL_DV = 256, COL_DK = 256 + D_;
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

constexpr uint32_t kErrMisaligned = 0x10u;

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void red_add_f32(float* addr, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity,
                                                uint64_t limit_ns) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity))
    if (globaltimer_ns() - t0 > limit_ns) return false;
  return true;
}

// Walk the query tiles (i, t) that see this CTA's KV tile, in the order of the schedule:
//   TO (tile-outer; striped layout only): t from the last tile down to the first visible
//     one, and for each t the query shards in ring order (in the striped layout query tile
//     t sees KV tile u of every shard iff t >= u);
//   otherwise the ring steps outermost, shard i = (j + k) mod P, and its visible query
//     tiles t_lo(i) .. T - 1 inside.
// f(i, t) handles one item and returns false to stop (a wait gave up).
template <bool TO, class F>
__device__ __forceinline__ bool bwd_walk(const BwdSched& sc, F&& f) {
  if (TO) {
    const int tmin = sc.t_lo(sc.j);
    for (int t = sc.T - 1; t >= tmin; --t)
      for (int k = 0; k < sc.P; ++k)
        if (!f(sc.i_of(k), t)) return false;
  } else {
    for (int k = 0; k < sc.P; ++k) {
      const int i = sc.i_of(k);
      for (int t = sc.t_lo(i); t < sc.T; ++t)
        if (!f(i, t)) return false;
    }
  }
  return true;
}

template <int D_, bool TO>
__global__ void __launch_bounds__(640, 1)
    ra_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                  const BwdArgs a) {
  using C = BwdCfg<D_>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* sm = smem_raw;
  uint8_t* sK = sm + C::OFF_K;
  uint8_t* sV = sm + C::OFF_V;
  uint8_t* sQ = sm + C::OFF_Q;
  uint8_t* sDO = sm + C::OFF_DO;
  uint8_t* sDS = sm + C::OFF_DS;
  float* sLD = reinterpret_cast<float*>(sm + C::OFF_LD);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  uint64_t* kv_full = bars;
  uint64_t* q_full = bars + 1;
  uint64_t* q_empty = q_full + NSTQ;
  uint64_t* s_full = q_empty + NSTQ;
  uint64_t* ds_ready = s_full + 1;
  uint64_t* ds_free = ds_ready + 1;
  uint64_t* dq_full = ds_free + 1;
  uint64_t* dq_empty = dq_full + 1;
  uint64_t* kv_final = dq_empty + 1;
  uint64_t* drain = kv_final + 1;
  uint32_t* misc = reinterpret_cast<uint32_t*>(sm + C::OFF_MISC);
  uint32_t* tmem_slot = misc;
  volatile uint32_t* abort_flag = misc + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // The 128-byte swizzle atoms need a 1024-byte aligned base; this kernel carries no
  // slack to realign, so a misaligned base is reported (error word) instead of used.
  if ((smem_u32(smem_raw) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicOr(a.err, kErrMisaligned);
    return;
  }

  // ---- decode: one (batch, key/value head) after another (the resident CTAs then share
  // its query heads' Q, dO and dQ accumulator in L2); inside it, heavy KV tiles first ---
  const int per_bh = a.P * a.T;
  const int bh = blockIdx.x / per_bh;
  const int idx = blockIdx.x % per_bh;
  int j, u;
  if (a.layout == RA_LAYOUT_STRIPED || !a.causal) {
    // consecutive CTAs: the same KV tile u (the same work) of every shard j, heaviest
    // (smallest u) first.  With the tile-outer walk such a group runs in step and reads the
    // same query tile row of every shard within P items of each other, so one L2 fill of
    // Q, dO and the dQ rows serves the group.
    u = idx / a.P;
    j = idx % a.P;
  } else if (a.layout == RA_LAYOUT_ZIGZAG) {
    // idx = natural-order position of the KV tile (smallest first = most query tiles)
    const int th = a.T >> 1, ch = idx / th;
    j = ch < a.P ? ch : 2 * a.P - 1 - ch;
    u = idx % th + (ch < a.P ? 0 : th);
  } else {
    j = idx / a.T;
    u = idx % a.T;
  }
  const int b = bh / a.Hkv, hk = bh % a.Hkv;
  const BwdSched sc{j, u, a.n, a.T, a.P, a.layout, a.causal};

  if (threadIdx.x == 0) {
    *abort_flag = (*(volatile unsigned int*)a.err != 0u) ? 1u : 0u;
    mbar_init(kv_full, 1);
    for (int st = 0; st < NSTQ; ++st) {
      mbar_init(&q_full[st], 1);
      mbar_init(&q_empty[st], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(ds_ready, 256);
    mbar_init(ds_free, 1);
    mbar_init(dq_full, 1);
    mbar_init(dq_empty, 256);
    mbar_init(kv_final, 1);
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if constexpr (D_ < 128) {
    // K's feature columns [D_, 128): zero for the dQ^T product (no TMA writes there)
    uint4* pad = reinterpret_cast<uint4*>(sK + (D_ / 64) * kTile * 128);
    for (int x = threadIdx.x; x < ((128 - D_) / 64) * kTile * 128 / 16; x += blockDim.x)
      pad[x] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
  }
  __syncthreads();
  if (*abort_flag) return;   // an earlier CTA gave up: uniform early exit, nothing held
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const WaitCtx wc{abort_flag, a.err, a.wait_limit_ns};
  const size_t ld_base = (size_t)b * a.H * a.L;   // [B, H, P, n] shard-major arrays

  if (warp == 0) {
    // ================================================================ producer =====
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmDO);
      mbar_expect_tx(kv_full, 2 * C::VB);
      for (int cb = 0; cb < D_ / 64; ++cb) {
        if (!check(a.err, rows_box_ok(cb * 64, hk, j, u * kTile, b, a.n, a.P, a.Hkv, a.B, D_),
                   kChkTma))
          continue;
        load_rows(sK + cb * kTile * 128, &tmK, kv_full, a.layout, cb * 64, hk, j, u * kTile, b,
                  a.n, a.P);
        load_rows(sV + cb * kTile * 128, &tmV, kv_full, a.layout, cb * 64, hk, j, u * kTile, b,
                  a.n, a.P);
      }
      int m = 0;
      bool ok = true;
      for (int g = 0; g < a.G && ok; ++g) {
        const int h = hk * a.G + g;
        ok = bwd_walk<TO>(sc, [&](int i, int t) -> bool {
            const int st = m % NSTQ;
            if (m >= NSTQ && !mbar_wait(&q_empty[st], ((m / NSTQ) - 1) & 1, wc)) return false;
            mbar_expect_tx(&q_full[st], 2 * C::QB + C::LDB);
            const size_t off = ld_base + (size_t)h * a.L + (size_t)i * a.n + (size_t)t * BQ;
            if (check(a.err, rows_box_ok(0, h, i, t * BQ, b, a.n, a.P, a.H, a.B, D_) &&
                                 off + BQ <= (size_t)a.B * a.H * a.L && st < NSTQ,
                      kChkTma)) {
              for (int cb = 0; cb < D_ / 64; ++cb) {
                load_rows(sQ + st * C::QB + cb * BQ * 128, &tmQ, &q_full[st], a.layout, cb * 64,
                          h, i, t * BQ, b, a.n, a.P);
                load_rows(sDO + st * C::QB + cb * BQ * 128, &tmDO, &q_full[st], a.layout,
                          cb * 64, h, i, t * BQ, b, a.n, a.P);
              }
              bulk_load(sLD + st * (2 * BQ), a.lse + off, BQ * 4, &q_full[st]);
              bulk_load(sLD + st * (2 * BQ) + BQ, a.Dvec + off, BQ * 4, &q_full[st]);
            }
            ++m;
            return true;
        });
      }
      if (kChecked) misc[2] = m;                 // items loaded, compared at the exit
      // let every copy this thread issued land before the CTA can exit
      mbar_wait_drain(kv_full, 0, a.wait_limit_ns);
      for (int r = (m > NSTQ ? m - NSTQ : 0); r < m; ++r)
        mbar_wait_drain(&q_full[r % NSTQ], (r / NSTQ) & 1, a.wait_limit_ns);
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer ===
    {  // the whole warp; one elected lane issues
      constexpr uint32_t idKK = idesc_bf16(128, 128, false, false);   // S^T, dP^T
      constexpr uint32_t idKM = idesc_bf16(128, D_, false, true);     // dV, dK
      constexpr uint32_t idMM = idesc_bf16(128, BQ, true, true);      // dQ^T
      const uint32_t k_addr = smem_u32(sK), v_addr = smem_u32(sV);
      const uint32_t q_addr = smem_u32(sQ), do_addr = smem_u32(sDO);
      const uint32_t ds_addr = smem_u32(sDS);
      const uint32_t tS = tbase + C::COL_S, tDP = tbase + C::COL_DP;
      const uint32_t tDV = tbase + C::COL_DV, tDK = tbase + C::COL_DK;
      // base descriptors; per-MMA offsets are added in 16-byte units
      const uint64_t kK = sdesc_kmajor(k_addr), vK = sdesc_kmajor(v_addr);
      const uint64_t kMN = sdesc_mnmajor(k_addr, kTile * 128);     // K^T: M = features
      const uint64_t dsK = sdesc_kmajor(ds_addr);                  // dS^T: rows = keys
      const uint64_t dsMN = sdesc_mnmajor(ds_addr, kTile * 128);   // dS^T: N = queries
      bool ok = mbar_wait_w(kv_full, 0, wc);
      tc_fence_after();
      // S^T, dP^T, dV and dK inside the allocation and disjoint
      if (!check(a.err, C::COL_S + 128 <= C::COL_DP && C::COL_DP + 128 <= C::COL_DV &&
                            C::COL_DV + D_ <= C::COL_DK && C::COL_DK + D_ <= 512, kChkTmem))
        ok = false;
      int total = 0;
      for (int k = 0; k < a.P; ++k) total += sc.T - sc.t_lo(sc.i_of(k));
      total *= a.G;

      // scores: A = K or V (K-major, 128 keys), B = Q or dO tile (K-major), K = D
#define RA_SCORES(D_TM, AK, BADDR)                                                        \
  do {                                                                                    \
    const uint64_t bd_ = sdesc_kmajor(BADDR);                                             \
    _Pragma("unroll") for (int kk = 0; kk < D_ / 16; ++kk) {                              \
      const uint32_t off = ((kk / 4) * (kTile * 128) + (kk % 4) * 32) >> 4;               \
      umma_ss_w(D_TM, (AK) + off, bd_ + off, idKK, kk > 0 ? 1u : 0u);                       \
    }                                                                                     \
  } while (0)

      if (ok && total > 0) {
        ok = mbar_wait_w(&q_full[0], 0, wc);
        tc_fence_after();
        if (ok) {
          RA_SCORES(tS, kK, q_addr);
          RA_SCORES(tDP, vK, do_addr);
          umma_commit_w(s_full);
        }
      }
      for (int m = 0; m < total && ok; ++m) {
        const int st = m % NSTQ, st1 = (m + 1) % NSTQ;
        const uint32_t qa = q_addr + st * C::QB, da = do_addr + st * C::QB;
        // the next Q/dO stage (loaded long before) is tested while the score warps still
        // work, inside the wait below rather than between products
        if (m + 1 < total && !mbar_wait_w(&q_full[st1], ((m + 1) / NSTQ) & 1, wc)) { ok = false; break; }
        if (!mbar_wait_w(ds_ready, m & 1, wc)) { ok = false; break; }
        tc_fence_after();
        // dQ^T = K^T dS^T into the dP region (dP^T(m) already consumed)   (K = 128 keys);
        // first, so that the drain warps can start on it while dV and S^T(m+1) run
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          umma_ss_w(tDP, kMN + ((kk * 2048) >> 4), dsMN + ((kk * 2048) >> 4), idMM,
                  kk > 0 ? 1u : 0u);
        umma_commit_w(dq_full);
        // dV += P^T dO   (K = 128 query rows; P^T is read from TMEM: warpgroup g left the
        // bf16 pairs of query columns [64g, 64g+64) in TMEM columns [64g, 64g+32))
        {
          const uint64_t bd = sdesc_mnmajor(da, BQ * 128);
#pragma unroll
          for (int kk = 0; kk < BQ / 16; ++kk)
            umma_ts_w(tDV, tS + (kk / 4) * 64 + (kk % 4) * 8, bd + ((kk * 2048) >> 4), idKM,
                    (m > 0 || kk > 0) ? 1u : 0u);
        }
        if (m + 1 < total) {
          // S^T(m+1): the S region is free once dV(m) has read P^T(m) (in-order pipe)
          RA_SCORES(tS, kK, q_addr + st1 * C::QB);
          // dP^T(m+1) once the drain warps have read dQ^T(m) out of the dP region
          if (!mbar_wait_w(dq_empty, m & 1, wc)) { ok = false; break; }
          tc_fence_after();
          RA_SCORES(tDP, vK, do_addr + st1 * C::QB);
          umma_commit_w(s_full);
        }
        // dK += dS^T Q   (K = 128 query rows); runs under the next tile's score work
        {
          const uint64_t bd = sdesc_mnmajor(qa, BQ * 128);
#pragma unroll
          for (int kk = 0; kk < BQ / 16; ++kk) {
            const uint32_t offa = ((kk / 4) * (kTile * 128) + (kk % 4) * 32) >> 4;
            umma_ss_w(tDK, dsK + offa, bd + ((kk * 2048) >> 4), idKM, (m > 0 || kk > 0) ? 1u : 0u);
          }
        }
        umma_commit_w(ds_free);       // dS^T(m) read by dQ^T(m) and dK(m)
        umma_commit_w(&q_empty[st]);  // Q(m), dO(m) read for the last time
      }
#undef RA_SCORES
      if (kChecked && lane == 0) misc[3] = total;             // compared at the exit
      umma_commit_w(kv_final);
      umma_commit_w(drain);
      if (!ok) mbar_wait_drain(drain, 0, a.wait_limit_ns);
    }
  } else if (warp >= 4 && warp < 12) {
    // ================================================================ key rows =====
    const int wq = warp & 3;
    const int half = (warp - 4) >> 2;             // query columns [64*half, 64*half + 64)
    const int brow = wq * 32 + lane;              // key row
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tbase + lane_off + C::COL_S + 64 * half;
    const uint32_t tDP = tbase + lane_off + C::COL_DP + 64 * half;
    const float sl2 = a.scale_log2;
    uint8_t* drow = sDS + half * (kTile * 128) + brow * 128;
    // this thread's S^T, dP^T columns and its dS^T row: inside the allocation, the warp's
    // lane quarter and the dS^T tile
    bool ok = check(a.err, tmem_ok(tS, tbase, 64, warp) && tmem_ok(tDP, tbase, 64, warp) &&
                               drow + 128 <= sDS + C::SB, kChkTmem | kChkSmem);
    int m = 0;
    for (int g = 0; g < a.G && ok; ++g) {
      ok = bwd_walk<TO>(sc, [&](int i, int t) -> bool {
          const int st = m % NSTQ;
          if (!mbar_wait(s_full, m & 1, wc) || !mbar_wait(&q_full[st], (m / NSTQ) & 1, wc))
            return false;
          // dS^T(m) overwrites the shared tile once dQ^T(m-1) and dK(m-1) have read it
          if (m >= 1 && !mbar_wait(ds_free, (m - 1) & 1, wc)) return false;
          tc_fence_after();
          const float* lse2 = sLD + st * (2 * BQ) + 64 * half;   // -lse * log2(e)
          const float* dvec = lse2 + BQ;                          // -D
          const long long dl = a.causal ? sc.delta(i, t) : (1LL << 40);
          // visible iff col - brow + delta >= 0 with col = 64*half + c, i.e. c >= lim
          const long long lim = (long long)brow - dl - 64 * half;
          // four passes of 16 query columns; pass p writes its P^T pairs to TMEM columns
          // [64*half + 8p, +8), inside S^T columns this warpgroup has already read.
          // Column pairs go through the packed fp32x2 FMA pipe: x = s*c + (-lse2),
          // dS = P * (dP + (-D)); the mask is applied only on tiles that need one.
          const bool masked = __any_sync(0xffffffffu, lim > 0);   // whole warp votes
          const uint64_t c2 = f2_pack(sl2, sl2);
#pragma unroll
          for (int pass = 0; pass < 4; ++pass) {
            uint32_t sr[16], pr[16];
            tmem_ld16(tS + 16 * pass, sr);
            tmem_ld16(tDP + 16 * pass, pr);
            tmem_wait_ld();
            uint32_t pw[8], dw[8];
#pragma unroll
            for (int g8 = 0; g8 < 2; ++g8) {
              const int cb = 16 * pass + 8 * g8;      // first of 8 columns
              // negated lse2 and D of the 8 columns, as 4 packed pairs each
              const ulonglong2 l01 = *reinterpret_cast<const ulonglong2*>(lse2 + cb);
              const ulonglong2 l23 = *reinterpret_cast<const ulonglong2*>(lse2 + cb + 4);
              const ulonglong2 d01 = *reinterpret_cast<const ulonglong2*>(dvec + cb);
              const ulonglong2 d23 = *reinterpret_cast<const ulonglong2*>(dvec + cb + 4);
              const uint64_t nl[4] = {l01.x, l01.y, l23.x, l23.y};
              const uint64_t nd[4] = {d01.x, d01.y, d23.x, d23.y};
#pragma unroll
              for (int e2 = 0; e2 < 4; ++e2) {
                const int c = cb + 2 * e2;
                const uint64_t s2 = f2_pack(__uint_as_float(sr[8 * g8 + 2 * e2]),
                                            __uint_as_float(sr[8 * g8 + 2 * e2 + 1]));
                const uint64_t dp2 = f2_pack(__uint_as_float(pr[8 * g8 + 2 * e2]),
                                             __uint_as_float(pr[8 * g8 + 2 * e2 + 1]));
                float x0, x1;
                f2_unpack(f2_fma(s2, c2, nl[e2]), x0, x1);
                float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                if (masked) {
                  if ((long long)c < lim) p0 = 0.f;
                  if ((long long)c + 1 < lim) p1 = 0.f;
                }
                const uint64_t pp2 = f2_pack(p0, p1);
                float ds0, ds1;
                f2_unpack(f2_mul(pp2, f2_add(dp2, nd[e2])), ds0, ds1);
                pw[4 * g8 + e2] = pack_bf16x2(p0, p1);
                dw[4 * g8 + e2] = pack_bf16x2(ds0, ds1);
              }
            }
            tmem_st8(tbase + lane_off + C::COL_S + 64 * half + 8 * pass, pw);
#pragma unroll
            for (int g8 = 0; g8 < 2; ++g8) {
              const int c8 = 2 * pass + g8;           // 16-byte chunk inside the 128-byte row
              *reinterpret_cast<uint4*>(drow + ((c8 ^ (brow & 7)) * 16)) =
                  make_uint4(dw[4 * g8], dw[4 * g8 + 1], dw[4 * g8 + 2], dw[4 * g8 + 3]);
            }
          }
          fence_proxy_async_smem();
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(ds_ready);
          ++m;
          return true;
      });
    }
    if (kChecked && brow == 0) misc[4 + half] = m;   // compared at the exit
    // ---- dK, dV epilogue (thread = key row): warpgroup 0 writes dV, 1 writes dK ------
    if (ok && mbar_wait(kv_final, 0, wc)) {
      tc_fence_after();
      const int loc = u * kTile + brow;
      const long long tok = token_of(a.layout, j, loc, a.n, a.P);
      const size_t row = ((size_t)b * a.L + tok) * a.Hkv + hk;
      const bool any = m > 0;
      const uint32_t tcol = tbase + lane_off + (half ? C::COL_DK : C::COL_DV);
      const float mul = half ? a.scale : 1.f;
      __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(half ? a.dk : a.dv) + row * D_;
      const bool in_range = check(a.err, tok >= 0 && tok < a.L && row < (size_t)a.B * a.L * a.Hkv &&
                                             tmem_ok(tcol, tbase, D_, warp),
                                  kChkGlobal);
#pragma unroll
      for (int c = 0; c < (in_range ? D_ / 32 : 0); ++c) {
        uint32_t r[32];
        tmem_ld32(tcol + 32 * c, r);
        tmem_wait_ld();
        uint4* o = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float f[8];
#pragma unroll
          for (int x = 0; x < 8; ++x) f[x] = any ? __uint_as_float(r[8 * e + x]) * mul : 0.f;
          o[e] = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                            pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
        }
      }
    }
  } else if (warp >= 12) {
    // ================================================================ dQ drain =====
    // thread = feature row d (TMEM lane), warpgroup g takes query columns [64g, 64g+64)
    const int wq = warp & 3;
    const int half = (warp - 12) >> 2;
    const int drow = wq * 32 + lane;
    const uint32_t tQ = tbase + (static_cast<uint32_t>(wq * 32) << 16) + C::COL_DP + 64 * half;
    const long long qstride = (a.layout == RA_LAYOUT_STRIPED) ? (long long)a.P * a.H * D_
                                                              : (long long)a.H * D_;
    bool ok = check(a.err, tmem_ok(tQ, tbase, 64, warp), kChkTmem);
    int m = 0;
    for (int g = 0; g < a.G && ok; ++g) {
      float* dq_head =
          a.dq_acc + (size_t)b * a.L * a.H * D_ + (size_t)(hk * a.G + g) * D_ + drow;
      ok = bwd_walk<TO>(sc, [&](int i, int t) -> bool {
          if (!mbar_wait(dq_full, m & 1, wc)) return false;
          tc_fence_after();
          uint32_t q0[32], q1[32];
          tmem_ld32(tQ, q0);
          tmem_ld32(tQ + 32, q1);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(dq_empty);
          ++m;
          if (drow >= D_) return true;   // a zero row of the padded K (D_ = 64)
          // 64 consecutive local rows: consecutive tokens (stride qstride) in every layout
          const long long tok0 = token_of(a.layout, i, t * BQ + 64 * half, a.n, a.P);
          float* p0 = dq_head + tok0 * a.H * D_;
          // the 64 rows' elements inside the accumulator (first and last token, the head)
          if (!check(a.err, tok0 >= 0 && tok0 + 63 * (qstride / (a.H * D_)) < a.L &&
                                hk * a.G + g < a.H &&
                                token_of(a.layout, i, t * BQ + 64 * half + 63, a.n, a.P) ==
                                    tok0 + 63 * (qstride / (a.H * D_)),
                     kChkGlobal))
            return true;
#pragma unroll
          for (int c = 0; c < 32; ++c) red_add_f32(p0 + c * qstride, __uint_as_float(q0[c]));
#pragma unroll
          for (int c = 0; c < 32; ++c) red_add_f32(p0 + (32 + c) * qstride, __uint_as_float(q1[c]));
          return true;
      });
    }
    if (kChecked && drow == 0) misc[6 + half] = m;   // compared at the exit
  }

  tc_fence_before();
  __syncthreads();
  if (kChecked && threadIdx.x == 0 && !*abort_flag)
    // the producer, the MMA issuer, both key-row and both drain warpgroups walked the
    // same number of query tiles
    check(a.err, misc[2] == misc[3] && misc[4] == misc[3] && misc[5] == misc[3] &&
                     misc[6] == misc[3] && misc[7] == misc[3], kChkSched);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

}  // namespace

template <int D_, bool TO>
cudaError_t launch_bwd_d(const BwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                         const CUtensorMap& tv, const CUtensorMap& tdo, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(ra_bwd_kernel<D_, TO>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       BwdCfg<D_>::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)a.B * a.Hkv * a.P * a.T;
  if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  ra_bwd_kernel<D_, TO><<<(unsigned)grid, 640, BwdCfg<D_>::SMEM_BYTES, s>>>(tq, tk, tv, tdo, a);
  return cudaGetLastError();
}

cudaError_t launch_bwd(const BwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const CUtensorMap& tdo, cudaStream_t s) {
  // tile-outer walk for the striped layout once a head's Q, dO and fp32 dQ accumulator
  // outgrow half the L2 (there the default order re-reads them from DRAM)
  const bool to = a.layout == RA_LAYOUT_STRIPED &&
                  8.0 * (double)a.L * a.D >= (double)kTileOuterBytes;
  if (a.D == 128) return to ? launch_bwd_d<128, true>(a, tq, tk, tv, tdo, s)
                            : launch_bwd_d<128, false>(a, tq, tk, tv, tdo, s);
  if (a.D == 64) return to ? launch_bwd_d<64, true>(a, tq, tk, tv, tdo, s)
                           : launch_bwd_d<64, false>(a, tq, tk, tv, tdo, s);
  return cudaErrorNotSupported;
}

}  // namespace ra
