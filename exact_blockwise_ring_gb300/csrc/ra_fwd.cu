// ra_fwd.cu -- forward kernel of exact blockwise ring attention on tcgen05 tensor cores.
//
// Method (labhub "Ring Attention 論文分析"):
//   * blockwise attention with an online softmax, section "ブロック単位の分割戦略":
//     per KV block, new_max = max(max, blockmax), correction = exp(max - new_max),
//     sum = sum * correction + rowsum(exp(s - new_max)), acc = acc * correction + P V;
//     finally out = acc / sum;
//   * ring order, section "リングトポロジーと KV の循環" (and the vanos001 ring diagram):
//     the queries of shard i visit KV shards (i - k) mod P for k = 0..P-1 (for the
//     striped layout at sizes where a head's K and V exceed half the L2, tile index by
//     tile index: for u = 0, 1, ..., the ring's shards in that order; CTAs launched side
//     by side then read each K/V tile row within a few items of each other, so one DRAM
//     fill serves them: at a million tokens a head's K and V are several times the L2);
//   * causal skipping, section "Causal Masking の処理": KV tiles after the query tile
//     are skipped, the diagonal tile is masked, earlier tiles are not.
//
// One CTA owns 256 query rows of one (batch, head, shard): two 128-row tiles that share
// every K/V tile loaded.  With grouped-query attention query head h reads key/value head
// h / G; CTAs run head after head, so the G query heads of a group, which read the same
// K/V, are adjacent in launch order and share those tiles in L2.  Roles (384 threads):
//   warp 0      TMA producer of Q (once) and of the K tiles (NK-stage ring)
//   warp 1      TMEM allocator and tcgen05.mma issuer: the whole warp walks the issue
//               loop (descriptors stay warp-uniform) and one elected lane issues
//   warp 2      per-shard work counter (one thread), otherwise idle
//   warp 3      TMA producer of the V tiles (NV-stage ring); both producer warps walk
//               their loops as whole warps, one elected lane issuing the copies
//   warps 4-7   softmax of query tile 0 (thread = query row = TMEM lane)
//   warps 8-11  softmax of query tile 1
// TMEM columns: S0/P0 [0,128), S1/P1 [128,256), O0 [256,256+D), O1 [256+D,256+2D).
// P (bf16) overwrites the low half of its S columns and is the TMEM A operand of P V.
// MMA issue order per KV tile n: PV0(n-1), S0(n), PV1(n-1), S1(n), so each softmax
// warpgroup overlaps the other tile's two MMAs.  K and V have separate rings: a K tile is
// released as soon as both S MMAs that read it are done, a V tile after both PV MMAs.
//
// Online-softmax details: exponentials are taken in base 2 with the running max m kept in
// raw score units, P = exp2((s - m) * scale * log2 e), so the maximum element gets exactly
// 1; m is refreshed only when a new tile max exceeds it by more than kTau in the log2
// domain (2^8 headroom), which is exact because the final normalisation and lse use the
// same stale max.  A row that has seen no visible key keeps max = -inf and
// takes P = 0 (the -inf guard).  The row sum accumulates fp32 P before P is rounded to
// bf16 for the tensor core.
#include <cuda_bf16.h>

#include "ra_check.cuh"
#include "ra_exp2.cuh"
#include "ra_internal.h"
#include "ra_ptx.cuh"
#include "ra_rows.cuh"

namespace ra {

namespace {

constexpr float kTau = 8.0f;
// One column pair in every kSoftExpEvery takes its exponentials in software on the FMA
// pipe (ra_exp2.cuh) instead of the exponential unit, which the softmax keeps busy;
// 0 = all on the exponential unit.
constexpr int kSoftExpEvery = 0;
constexpr float kNegInf = -__builtin_huge_valf();

template <int D>
struct FwdCfg {
  static constexpr int NK = (D == 64) ? 4 : 3;        // K pipeline stages
  static constexpr int NV = (D == 64) ? 4 : 2;        // V pipeline stages
  static constexpr int QB = kTile * D * 2;            // bytes of one Q tile
  static constexpr int KVB = kTile * D * 2;           // bytes of one K or V tile
  static constexpr int NCB = D / 64;                  // 128-byte column blocks per row
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + 2 * QB;
  static constexpr int OFF_V = OFF_K + NK * KVB;
  static constexpr int OFF_BAR = OFF_V + NV * KVB;
  // barriers: q_full, k_full[NK], k_empty[NK], v_full[NV], v_empty[NV], s_full[2],
  //           p_full[2], o_final[2], drain
  static constexpr int NBAR = 1 + 2 * NK + 2 * NV + 7;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 64 + 1024;   // + 1024 alignment slack
  static constexpr int COL_S = 0;          // + 128 * q
  static constexpr int COL_O = 256;        // + D * q
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity,
                                                uint64_t limit_ns) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity))
    if (globaltimer_ns() - t0 > limit_ns) return false;
  return true;
}

// Work counter for one CTA and its ring steps (closed forms of the tiles it visits).
__device__ void count_work(const FwdArgs& a, const RingSched& sc, int g) {
  unsigned long long* tiles = a.shard_work;
  unsigned long long* pairs = a.shard_work + a.P;
  unsigned long long* visits = a.shard_work + 2 * a.P;
  const int i = sc.i;
  const int Tb = a.n / a.block;
  unsigned long long n_tiles = 0, n_pairs = 0;
  // query blocks of `block` rows owned by this CTA: rows [128*t0, 128*(t0+nq)) clipped
  const int r0 = kTile * sc.t0;
  int r1 = kTile * (sc.t0 + sc.nq);
  if (r1 > a.n) r1 = a.n;
  for (int k = sc.k0; k < sc.k1; ++k) {
    const int j = sc.j_of(k);
    for (int tb = r0 / a.block; tb * a.block < r1; ++tb) {
      if (!a.causal) n_tiles += Tb;
      else if (a.layout == RA_LAYOUT_STRIPED) n_tiles += tb + 1;
      else n_tiles += blocks_upto(a.layout, j, block_pos(a.layout, i, tb, Tb, a.P), Tb, a.P);
    }
    const unsigned long long R = r1 - r0;
    const unsigned long long sum_a = R * r0 + R * (R - 1) / 2;   // sum of local rows a
    if (!a.causal) n_pairs += R * a.n;
    else if (a.layout == RA_LAYOUT_STRIPED) n_pairs += (j <= i) ? sum_a + R : sum_a;
    else if (a.layout == RA_LAYOUT_CONTIGUOUS)
      n_pairs += (j < i) ? R * a.n : (j == i ? sum_a + R : 0ull);
    else   // zigzag: row by row
      for (int r = r0; r < r1; ++r)
        n_pairs += tokens_upto(a.layout, j, token_of(a.layout, i, r, a.n, a.P), a.n, a.P);
  }
  atomicAdd(&tiles[i], n_tiles);
  atomicAdd(&pairs[i], n_pairs);
  if (g == 0) {
    unsigned long long v = 0;
    for (int r = r0; r < r1; ++r) {
      const long long tok = token_of(a.layout, i, r, a.n, a.P);
      v += a.causal ? (unsigned long long)(tok / a.block + 1)
                    : (unsigned long long)(a.L / a.block);
    }
    atomicAdd(&visits[i], v);
  }
}

// TO (tile-outer; striped layout only): every role walks KV tile index u outermost and
// the ring steps inside.  Otherwise the ring steps are outermost and the KV tiles of a
// step inside.
template <int D, bool TO>
__global__ void __launch_bounds__(384, 1)
    ra_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const FwdArgs a) {
  using C = FwdCfg<D>;
  constexpr int NK = C::NK, NV = C::NV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = sm + C::OFF_Q;
  uint8_t* sK = sm + C::OFF_K;
  uint8_t* sV = sm + C::OFF_V;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + NK;
  uint64_t* v_full = k_empty + NK;
  uint64_t* v_empty = v_full + NV;
  uint64_t* s_full = v_empty + NV;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_final = p_full + 2;
  uint64_t* drain = o_final + 2;
  uint32_t* misc = reinterpret_cast<uint32_t*>(sm + C::OFF_MISC);
  uint32_t* tmem_slot = misc;
  volatile uint32_t* abort_flag = misc + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- decode this CTA: one (batch, head) after another so that the CTAs resident at
  // any time share that head's K/V in L2; inside a head, heavy work first (for the
  // blocked layouts: tile pairs in descending natural-order position) ------------------
  const int per_bh = a.n_split * a.P * a.npair;
  const int bh = blockIdx.x / per_bh;
  int idx = blockIdx.x % per_bh;
  const int g = idx % a.n_split;
  idx /= a.n_split;
  int i, s;
  if (a.causal && a.layout == RA_LAYOUT_CONTIGUOUS) {
    const int pos = a.P * a.npair - 1 - idx;
    i = pos / a.npair;
    s = pos % a.npair;
  } else if (a.causal && a.layout == RA_LAYOUT_ZIGZAG && (a.T & 3) == 0) {
    // T/2 tiles per chunk, an even number: T/4 pairs per chunk, none straddles two
    const int hp = a.T >> 2;
    const int pos = a.P * a.npair - 1 - idx;
    const int ch = pos / hp;
    i = ch < a.P ? ch : 2 * a.P - 1 - ch;
    s = (ch < a.P ? 0 : hp) + pos % hp;
  } else {
    // consecutive CTAs: the same tile pair s (the same work) of every shard i, heaviest
    // first.  With the tile-outer walk such a group runs in step and reads the same KV tile
    // row of every shard within P items of each other, so one L2 fill serves the group.
    s = a.npair - 1 - idx / a.P;
    i = idx % a.P;
  }
  const int b = bh / a.H, h = bh % a.H;
  const int hkv = h / a.G;        // key/value head of this query head
  const int steps = a.P / a.n_split;
  RingSched sc{i, 2 * s, 2, a.T, a.P, a.layout, a.causal, g * steps, (g + 1) * steps};
  const int nvalid = (2 * s + 1 < a.T) ? 2 : 1;
  // Every role walks the same items, (u, j) pairs with a visible key for either query tile:
  //   ring steps outermost (KV shard j = (i - k) mod P), then u = 0 .. u_end(j) - 1; or
  //   (TO, striped) u = 0 .. umax - 1 outermost, then the ring steps in ring order; in the
  //   striped layout query tile t sees KV tiles u <= t of every shard (u == t masked), so
  //   every (u, j) with u < umax is an item and each query tile's visible prefix is the
  //   same for all j.
  const int umax = sc.u_max();

  if (threadIdx.x == 0) {
    *abort_flag = (*(volatile unsigned int*)a.err != 0u) ? 1u : 0u;
    mbar_init(q_full, 1);
    for (int st = 0; st < NK; ++st) {
      mbar_init(&k_full[st], 1);
      mbar_init(&k_empty[st], 1);
    }
    for (int st = 0; st < NV; ++st) {
      mbar_init(&v_full[st], 1);
      mbar_init(&v_empty[st], 1);
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(&s_full[q], 1);
      mbar_init(&p_full[q], 128);
      mbar_init(&o_final[q], 1);
    }
    mbar_init(drain, 1);
    fence_mbar_init();
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

  if (warp == 0 || warp == 3) {
    // ================================================================ producers ====
    // warp 0: Q once, then K tiles; warp 3: V tiles.  Both walk the same item sequence.
    {  // the whole warp; one elected lane issues
      const bool is_k = warp == 0;
      const int NS = is_k ? NK : NV;
      uint64_t* full = is_k ? k_full : v_full;
      uint64_t* empty = is_k ? k_empty : v_empty;
      uint8_t* ring = is_k ? sK : sV;
      const CUtensorMap* tm = is_k ? &tmK : &tmV;
      tma_prefetch_desc(tm);
      if (is_k) {
        tma_prefetch_desc(&tmQ);
        mbar_expect_tx_w(q_full, nvalid * C::QB);
        for (int q = 0; q < nvalid; ++q)
          for (int cb = 0; cb < C::NCB; ++cb)
            if (check(a.err, rows_box_ok(cb * 64, h, i, (2 * s + q) * kTile, b, a.n, a.P, a.H,
                                         a.B, D), kChkTma))
              load_rows<true>(sQ + q * C::QB + cb * kTile * 128, &tmQ, q_full, a.layout, cb * 64, h,
                        i, (2 * s + q) * kTile, b, a.n, a.P);
      }
      int n = 0;
      bool ok = true;
      auto item = [&](int u, int j) {
        const int st = n % NS;
        if (n >= NS && !mbar_wait_w(&empty[st], ((n / NS) - 1) & 1, wc)) return false;
        mbar_expect_tx_w(&full[st], C::KVB);
        for (int cb = 0; cb < C::NCB; ++cb)
          if (check(a.err, rows_box_ok(cb * 64, hkv, j, u * kTile, b, a.n, a.P, a.H / a.G, a.B,
                                       D) && st < NS, kChkTma))
            load_rows<true>(ring + st * C::KVB + cb * kTile * 128, tm, &full[st], a.layout, cb * 64,
                      hkv, j, u * kTile, b, a.n, a.P);
        ++n;
        return true;
      };
      if (TO) {
        for (int u = 0; u < umax && ok; ++u)
          for (int kk = 0; kk < steps && ok; ++kk) ok = item(u, sc.j_of(sc.k0 + kk));
      } else {
        for (int kk = 0; kk < steps && ok; ++kk) {
          const int j = sc.j_of(sc.k0 + kk);
          const int ue = sc.u_end(j);
          for (int u = 0; u < ue && ok; ++u) ok = item(u, j);
        }
      }
      if (kChecked && lane == 0) misc[is_k ? 2 : 3] = n;     // items loaded, compared at the exit
      // let every copy this thread issued land before the CTA can exit
      if (is_k) mbar_wait_drain(q_full, 0, a.wait_limit_ns);
      for (int m = (n > NS ? n - NS : 0); m < n; ++m)
        mbar_wait_drain(&full[m % NS], (m / NS) & 1, a.wait_limit_ns);
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer ===
    {  // the whole warp; one elected lane issues
      constexpr uint32_t idS = idesc_bf16(128, 128, false, false);
      constexpr uint32_t idPV = idesc_bf16(128, D, false, true);
      const uint32_t q_addr = smem_u32(sQ), k_addr = smem_u32(sK), v_addr = smem_u32(sV);
      // per query tile: V stage / phase of the item whose PV is still to be issued (-1:
      // none) and the number of PVs issued so far; scalars, so nothing goes to local memory
      int pend0 = -1, pend1 = -1;
      uint32_t ppar0 = 0, ppar1 = 0;
      int pv0 = 0, pv1 = 0;
      bool ok = mbar_wait_w(q_full, 0, wc);
      tc_fence_after();
      const uint64_t q0d = sdesc_kmajor(q_addr), q1d = sdesc_kmajor(q_addr + C::QB);
      const uint32_t dS0 = tbase + C::COL_S, dS1 = tbase + C::COL_S + 128;
      const uint32_t dO0 = tbase + C::COL_O, dO1 = tbase + C::COL_O + D;
      // the four accumulators inside the allocation, S columns disjoint from O columns
      if (!check(a.err, C::COL_S + 256 <= C::COL_O && C::COL_O + 2 * D <= 512, kChkTmem))
        ok = false;
      int n_s0 = 0, n_s1 = 0;

#define RA_ISSUE_PV(PEND, PPAR, PV, PFULL, DO_, AP_)                                          \
  do {                                                                                        \
    if ((!v_seen && !mbar_wait_w(&v_full[PEND], PPAR, wc)) || !mbar_wait_w(PFULL, (PV) & 1, wc)) { \
      ok = false;                                                                             \
      break;                                                                                  \
    }                                                                                         \
    v_seen = true;                                                                            \
    tc_fence_after();                                                                         \
    const uint64_t vd = sdesc_mnmajor(v_addr + (PEND) * C::KVB, kTile * 128);                 \
    _Pragma("unroll") for (int kk = 0; kk < kTile / 16; ++kk)                                 \
        umma_ts_w(DO_, (AP_) + kk * 8, vd + ((kk * 2048) >> 4), idPV,                           \
                ((PV) > 0 || kk > 0) ? 1u : 0u);                                              \
    ++(PV);                                                                                   \
    (PEND) = -1;                                                                              \
  } while (0)

#define RA_ISSUE_S(QD, DS_)                                                                   \
  do {                                                                                        \
    _Pragma("unroll") for (int kk = 0; kk < D / 16; ++kk) {                                   \
      const uint32_t off = ((kk / 4) * (kTile * 128) + (kk % 4) * 32) >> 4;                   \
      umma_ss_w(DS_, (QD) + off, kd + off, idS, kk > 0 ? 1u : 0u);                              \
    }                                                                                         \
  } while (0)

      int n = 0;
      // one item: the S MMA of each query tile that sees KV tile u (u < ue_q), each after
      // the PV of that tile's previous item
      auto item = [&](int u, int ue0, int ue1) -> bool {
          const int kst = n % NK, vst = n % NV;
          // both PVs of this item use the previous item's V tile: wait for it once
          bool v_seen = false;
          if (!mbar_wait_w(&k_full[kst], (n / NK) & 1, wc)) return false;
          tc_fence_after();
          const uint64_t kd = sdesc_kmajor(k_addr + kst * C::KVB);
          // query tile 0
          if (pend0 >= 0) RA_ISSUE_PV(pend0, ppar0, pv0, &p_full[0], dO0, dS0);
          if (!ok) return false;
          if (!check(a.err, kst < NK && vst < NV, kChkSmem)) return false;
          if (u < ue0) {
            RA_ISSUE_S(q0d, dS0);
            ++n_s0;
            umma_commit_w(&s_full[0]);
            pend0 = vst;
            ppar0 = (n / NV) & 1;
          }
          // query tile 1
          if (pend1 >= 0) RA_ISSUE_PV(pend1, ppar1, pv1, &p_full[1], dO1, dS1);
          if (!ok) return false;
          if (u < ue1) {
            RA_ISSUE_S(q1d, dS1);
            ++n_s1;
            umma_commit_w(&s_full[1]);
            pend1 = vst;
            ppar1 = (n / NV) & 1;
          }
          umma_commit_w(&k_empty[kst]);                       // both S MMAs of item n issued
          if (n > 0) umma_commit_w(&v_empty[(n - 1) % NV]);    // every PV of item n-1 issued
          ++n;
          return true;
      };
      if (TO) {
        // striped: each query tile sees the same prefix of every shard
        const int ue0 = sc.q_end(0, i), ue1 = sc.q_end(1, i);
        for (int u = 0; u < umax && ok; ++u)
          for (int kk = 0; kk < steps && ok; ++kk) ok = item(u, ue0, ue1);
      } else {
        for (int kk = 0; kk < steps && ok; ++kk) {
          const int j = sc.j_of(sc.k0 + kk);
          const int ue0 = sc.q_end(0, j), ue1 = sc.q_end(1, j);
          const int ue = ue0 > ue1 ? ue0 : ue1;
          for (int u = 0; u < ue && ok; ++u) ok = item(u, ue0, ue1);
        }
      }
      bool v_seen = false;
      if (ok && pend0 >= 0) RA_ISSUE_PV(pend0, ppar0, pv0, &p_full[0], dO0, dS0);
      if (ok && pend1 >= 0) RA_ISSUE_PV(pend1, ppar1, pv1, &p_full[1], dO1, dS1);
      if (ok && n > 0) umma_commit_w(&v_empty[(n - 1) % NV]);
#undef RA_ISSUE_PV
#undef RA_ISSUE_S
      if (kChecked && lane == 0) {              // compared at the exit
        misc[4] = n;
        misc[5] = n_s0;
        misc[6] = n_s1;
      }
      umma_commit_w(&o_final[0]);
      umma_commit_w(&o_final[1]);
      umma_commit_w(drain);
      if (!ok) mbar_wait_drain(drain, 0, a.wait_limit_ns);
    }
  } else if (warp == 2) {
    if (lane == 0 && a.shard_work != nullptr) count_work(a, sc, g);
  } else if (warp >= 4) {
    // ================================================================ softmax ======
    const int q = (warp - 4) >> 2;
    const int wq = warp & 3;
    const int arow = wq * 32 + lane;              // row inside the 128-row tile
    const int t = 2 * s + q;
    const bool valid = t < a.T;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tbase + lane_off + C::COL_S + q * 128;
    const uint32_t tO = tbase + lane_off + C::COL_O + q * D;
    const float sl2 = a.scale_log2;
    const float tau_raw = kTau / sl2;           // rescale threshold in raw score units
    float m_run = kNegInf, l_run = 0.f;         // running max (raw units) and row sum
    int cnt = 0;
    // this thread's S/P and O columns: inside the allocation and the warp's lane quarter
    bool ok = check(a.err, tmem_ok(tS, tbase, 128, warp) && tmem_ok(tO, tbase, D, warp),
                    kChkTmem);
    // one item: the scores of KV tile u of shard j (masked when on_diag)
    auto item = [&](bool on_diag, int j) -> bool {
          if (!mbar_wait(&s_full[q], cnt & 1, wc)) return false;
          tc_fence_after();
          // all four 32-column loads in flight before the one wait
          float sv[128];
          {
            uint32_t r0[32], r1[32], r2[32], r3[32];
            tmem_ld32(tS, r0);
            tmem_ld32(tS + 32, r1);
            tmem_ld32(tS + 64, r2);
            tmem_ld32(tS + 96, r3);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              sv[e] = __uint_as_float(r0[e]);
              sv[32 + e] = __uint_as_float(r1[e]);
              sv[64 + e] = __uint_as_float(r2[e]);
              sv[96 + e] = __uint_as_float(r3[e]);
            }
          }
          if (on_diag) {
            const int lim = arow - ((a.layout == RA_LAYOUT_STRIPED && j > i) ? 1 : 0);
#pragma unroll
            for (int e = 0; e < 128; ++e)
              if (e > lim) sv[e] = kNegInf;
          }
          float mx[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) mx[e] = fmaxf(sv[2 * e], sv[2 * e + 1]);   // sv[0..7]
#pragma unroll
          for (int e = 8; e < 128; e += 8) {                                       // sv[8..127]
            mx[0] = fmax3(mx[0], sv[e], sv[e + 1]);
            mx[1] = fmax3(mx[1], sv[e + 2], sv[e + 3]);
            mx[2] = fmax3(mx[2], sv[e + 4], sv[e + 5]);
            mx[3] = fmax3(mx[3], sv[e + 6], sv[e + 7]);
          }
          const float tmax = fmax3(fmax3(mx[0], mx[1], mx[2]), mx[3], mx[3]);
          // running max kept in raw score units: x = (s - m) * c is exactly 0 for the
          // maximum element, so a lone visible key gets P = 1 exactly
          const bool need = tmax > m_run + tau_raw;
          float corr = 1.f;
          if (need) {
            corr = ex2_approx((m_run - tmax) * sl2);
            l_run *= corr;
            m_run = tmax;
          }
          const float mu = (m_run == kNegInf) ? 0.f : m_run;
          // P = exp2((s - m) * c) two columns at a time: packed subtract and multiply, two
          // MUFU ex2, one packed add into the running row sum (two independent sum chains)
          const uint64_t c2 = f2_pack(sl2, sl2), nm2 = f2_pack(-mu, -mu);
          uint64_t acc2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              float x0, x1;
              f2_unpack(f2_mul(f2_add(f2_pack(sv[32 * c + 2 * e], sv[32 * c + 2 * e + 1]), nm2), c2),
                        x0, x1);
              float p0, p1;
              if (kSoftExpEvery > 0 && e % kSoftExpEvery == kSoftExpEvery - 1) {
                f2_unpack(exp2_soft_x2(x0, x1), p0, p1);     // on the FMA pipe
              } else {
                p0 = ex2_approx(x0);
                p1 = ex2_approx(x1);
              }
              acc2[e & 1] = f2_add(acc2[e & 1], f2_pack(p0, p1));
              pk[e] = pack_bf16x2(p0, p1);
            }
            tmem_st16(tS + 16 * c, pk);
          }
          {
            float a0, a1, b0, b1;
            f2_unpack(acc2[0], a0, a1);
            f2_unpack(acc2[1], b0, b1);
            l_run += (a0 + a1) + (b0 + b1);
          }
          // O *= correction (rare, lazy rescale), after the scores are no longer live; it
          // must land before P is published, because the next PV accumulates onto O
          if (cnt > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t r[32];
              tmem_ld32(tO + 32 * c, r);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * corr);
              tmem_st32(tO + 32 * c, r);
            }
          }
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&p_full[q]);
          ++cnt;
          return true;
    };
    if (valid) {
      if (TO) {
        // striped: the same visible prefix and diagonal tile in every shard
        const int ueq = sc.q_end(q, i), udiag = sc.q_diag(q, i);
        for (int u = 0; u < ueq && ok; ++u)
          for (int kk = 0; kk < steps; ++kk)
            if (!item(u == udiag, sc.j_of(sc.k0 + kk))) { ok = false; break; }
      } else {
        for (int kk = 0; kk < steps && ok; ++kk) {
          const int j = sc.j_of(sc.k0 + kk);
          const int ueq = sc.q_end(q, j), udiag = sc.q_diag(q, j);
          for (int u = 0; u < ueq; ++u) if (!item(u == udiag, j)) { ok = false; break; }
        }
      }
    }
    if (kChecked && arow == 0) misc[7 + q] = cnt;   // compared at the exit
    if (ok && mbar_wait(&o_final[q], 0, wc) && valid) {
      tc_fence_after();
      const int loc = t * kTile + arow;
      const long long tok = token_of(a.layout, i, loc, a.n, a.P);
      // l = 0: no visible key (out 0, lse -inf); a NaN row sum (a NaN input) stays NaN
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      const float lse_v =
          l_run == 0.f ? kNegInf : (m_run * sl2 + __log2f(l_run)) * 0.69314718055994531f;
      const size_t row = ((size_t)b * a.L + tok) * a.H + h;
      const size_t lidx = ((size_t)b * a.H + h) * a.L + tok;
      const bool in_range = check(
          a.err, tok >= 0 && tok < a.L && (row + 1) * D <= (size_t)a.B * a.L * a.H * D &&
                     lidx < (size_t)a.B * a.H * a.L && g < a.n_split,
          kChkGlobal);
      float* of32 = nullptr;
      __nv_bfloat16* obf = nullptr;
      if (in_range && a.n_split > 1) {
        of32 = a.o_part + (size_t)g * a.B * a.L * a.H * D + row * D;
        a.lse_part[(size_t)g * a.B * a.H * a.L + lidx] = lse_v;
      } else if (in_range) {
        if (a.out_fp32) of32 = reinterpret_cast<float*>(a.out) + row * D;
        else obf = reinterpret_cast<__nv_bfloat16*>(a.out) + row * D;
        a.lse[lidx] = lse_v;
      }
#pragma unroll
      for (int c = 0; c < (in_range ? D / 32 : 0); ++c) {
        uint32_t r[32];
        tmem_ld32(tO + 32 * c, r);
        tmem_wait_ld();
        if (of32) {
          float4* dst = reinterpret_cast<float4*>(of32 + 32 * c);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            dst[e] = make_float4(__uint_as_float(r[4 * e]) * inv, __uint_as_float(r[4 * e + 1]) * inv,
                                 __uint_as_float(r[4 * e + 2]) * inv,
                                 __uint_as_float(r[4 * e + 3]) * inv);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(obf + 32 * c);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(r[8 * e + 0]) * inv, __uint_as_float(r[8 * e + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(r[8 * e + 2]) * inv, __uint_as_float(r[8 * e + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(r[8 * e + 4]) * inv, __uint_as_float(r[8 * e + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(r[8 * e + 6]) * inv, __uint_as_float(r[8 * e + 7]) * inv);
            dst[e] = w;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (kChecked && threadIdx.x == 0 && !*abort_flag)
    // both producers and the MMA issuer walked the same items; each softmax warpgroup saw
    // as many score tiles as the MMA issuer computed for its query tile
    check(a.err, misc[2] == misc[3] && misc[3] == misc[4] && misc[5] == misc[7] &&
                     misc[6] == misc[8], kChkSched);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <int D, bool TO>
cudaError_t launch_fwd_d(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                         const CUtensorMap& tv, cudaStream_t st) {
  using C = FwdCfg<D>;
  cudaError_t e = cudaFuncSetAttribute(ra_fwd_kernel<D, TO>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)a.B * a.H * a.P * a.npair * a.n_split;
  if (grid <= 0 || grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  ra_fwd_kernel<D, TO><<<(unsigned)grid, 384, C::SMEM_BYTES, st>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const FwdArgs& a, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, cudaStream_t s) {
  // tile-outer walk for the striped layout once a key/value head's K and V outgrow half
  // the L2 (there the default order re-reads them from DRAM)
  const bool to = a.layout == RA_LAYOUT_STRIPED &&
                  4.0 * (double)a.L * a.D >= (double)kTileOuterBytes;
  if (a.D == 64) return to ? launch_fwd_d<64, true>(a, tq, tk, tv, s)
                           : launch_fwd_d<64, false>(a, tq, tk, tv, s);
  return to ? launch_fwd_d<128, true>(a, tq, tk, tv, s) : launch_fwd_d<128, false>(a, tq, tk, tv, s);
}

}  // namespace ra
