// prefill_bf16.cu -- bf16 attention forward on the 5th-generation tensor
// cores (tcgen05 + TMEM), sm_103a.
//
// What it computes is the FlashAttention-2 forward of the "FP32 CUDA-core
// FlashAttention-2 v2" blog (dandandamowang post_1787450400): Q blocks are
// resident for the whole KV loop (section 1.2), K/V blocks stream through a
// multi-stage buffer (section 3.2), the softmax is online with a deferred 1/l
// (sections 1.3, 3.3, 3.5), blocks above the causal diagonal are skipped and
// the block crossing it is masked per element (sections 1.4, 3.4).  P is cast
// to bf16 before the PV product, as item 7 of the FlashMLA issue #26 list
// suggests (fp32 -> bf16 conversion of P).
//
// How it maps onto GB300 (nothing here is taken from the pages' Ampere,
// Hopper or RTX kernels).  One CTA owns TWO consecutive 128-row Q tiles of
// one head and streams that head's K/V blocks once for both:
//   * warp 8  : TMA producer.  Both Q tiles once, then K_j and V_j together
//               into a ring of stages (128-byte swizzle), one full and one
//               empty mbarrier per stage.
//   * warp 9  : MMA issuer (one thread) and TMEM owner.  For tile t,
//               S_t = Q_t K_j^T (tcgen05.mma M=128 N=128 K=D) into TMEM, and
//               O_t += P_t V_j with P read straight from TMEM as the A operand,
//               in two halves of 64 keys.  The issue order S0_0, S1_0, PV0_0,
//               S0_1, PV1_0, S1_1, ... lets the tensor core work on one tile
//               while the other tile's softmax runs (ping-pong).
//   * warps 0-3 / 4-7 : softmax warpgroup of tile 0 / tile 1, one thread per
//               query row (TMEM lane = row).  Each block's 128 keys are taken
//               as two online-softmax steps of 64 keys: load the S half, mask,
//               exp2, row sum, write P (bf16) over already-read S columns and
//               hand that half to the MMA thread at once, so the PV of the
//               first half runs while the second half is computed.  The fast
//               path computes P with the current reference and no row max; it
//               is kept while every half-row sum is at most 2^16 (so every P
//               is), otherwise the half is redone with its exact max.  O in
//               TMEM is rescaled only when the max grew by more than 2^8 (lazy
//               rescale; exact because O and l share the stale reference), and
//               finally O/l -> bf16 -> smem -> TMA store, plus LSE.
//   TMEM columns: S0 [0,128), S1 [128,256), O0 [256,384), O1 [384,512).
//   Work order: heads in groups of 16 (the CTAs running together share those
//   heads' K/V in L2), heaviest causal Q pairs first within a group.
//   Every wait is bounded (about 2 s); a stuck pipeline records
//   ATTN_ERR_DEVICE_TIMEOUT and the CTA unwinds, frees TMEM and exits.
#include <math.h>

#include "common.cuh"

namespace {

using namespace gb300;

constexpr int kBM = 128;              // query rows per Q tile
constexpr int kBN = 128;              // keys per KV block
constexpr int kTilesPerCta = 2;
constexpr int kThreads = 320;         // 2 softmax warpgroups + producer + MMA
constexpr int kAtomBytes = 128 * 128; // one 128-row x 64-col bf16 swizzle column
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kFastSumLimit = 65536.0f;   // fast path kept while every half-row sum <= 2^16
constexpr int kHeadGroup = 16;             // heads scheduled together

template <int D>
struct Cfg {
  static constexpr int kAtoms = D / 64;
  static constexpr int kTileBytes = kAtoms * kAtomBytes;  // Q, K or V block
  static constexpr int kStageBytes = 2 * kTileBytes;      // K_j then V_j
  static constexpr int kStages = (D == 128) ? 2 : 5;      // ring slots (one KV block each)
  static constexpr int kQOff = 0;                          // Q0, Q1
  static constexpr int kRingOff = kTilesPerCta * kTileBytes;
  static constexpr int kBarOff = kRingOff + kStages * kStageBytes;
  // barriers: q_full, kv_full[S], kv_empty[S], s_full[tile], p_full[tile][half],
  // pv_done[tile][half], mma_drain.  The per-half barriers each complete once
  // per KV block, so no waiter is ever two phases behind or ahead of one.
  static constexpr int kNumBars = 1 + 2 * kStages + 2 + 4 + 4 + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // tmem base, abort flag
  static constexpr int kSmemBytes = kMiscOff + 16 + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;    // + 128 * tile
  static constexpr uint32_t kColO = 256;  // + 128 * tile
};

template <int D, bool kCausal>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_bf16_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV,
                        const __grid_constant__ CUtensorMap tmO, float* __restrict__ lse,
                        int BH, int N, float scale_log2, int* err, int debug_skip_load) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment: swizzle atoms must start on a 1024-byte boundary.
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);

  const uint32_t sQ = base + C::kQOff;
  const uint32_t sRing = base + C::kRingOff;
  const uint32_t bar0 = base + C::kBarOff;
  const uint32_t bar_q_full = bar0;
  auto bar_kv_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto bar_kv_empty = [&](int s) { return bar0 + 8u * (1 + C::kStages + s); };
  auto bar_s_full = [&](int t) { return bar0 + 8u * (1 + 2 * C::kStages + t); };
  auto bar_p_full = [&](int t, int h) { return bar0 + 8u * (3 + 2 * C::kStages + 2 * t + h); };
  auto bar_pv_done = [&](int t, int h) { return bar0 + 8u * (7 + 2 * C::kStages + 2 * t + h); };
  const uint32_t bar_mma_drain = bar0 + 8u * (11 + 2 * C::kStages);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work item: heads in groups of kHeadGroup (their K/V stay in L2);
  // within a group, heaviest causal Q pairs first across the group's heads.
  const int n_qt = (N + kBM - 1) / kBM;
  const int n_pairs = (n_qt + 1) / 2;
  const int group = blockIdx.x / (kHeadGroup * n_pairs);
  const int g_heads = min(kHeadGroup, BH - group * kHeadGroup);
  const int rem = blockIdx.x - group * kHeadGroup * n_pairs;
  const int bh = group * kHeadGroup + rem % g_heads;
  const int pr = kCausal ? (n_pairs - 1 - rem / g_heads) : (rem / g_heads);
  int Tt[kTilesPerCta];  // KV blocks visited by each Q tile (0: tile absent)
#pragma unroll
  for (int t = 0; t < kTilesPerCta; ++t) {
    const int qt = 2 * pr + t;
    if (qt >= n_qt) {
      Tt[t] = 0;
    } else {
      const int kv_limit = kCausal ? min(qt * kBM + kBM, N) : N;
      Tt[t] = (kv_limit + kBN - 1) / kBN;
    }
  }
  const int ntiles = Tt[1] > 0 ? 2 : 1;
  const int Tmax = max(Tt[0], Tt[1]);

  // ---- setup: barriers (thread 0), TMEM (warp 9)
  if (threadIdx.x == 0) {
    mbar_init(bar_q_full, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar_kv_full(s), 1);
      mbar_init(bar_kv_empty(s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar_s_full(t), 1);
      for (int h = 0; h < 2; ++h) {
        mbar_init(bar_p_full(t, h), 128);
        mbar_init(bar_pv_done(t, h), 1);
      }
    }
    mbar_init(bar_mma_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    prefetch_tmap(&tmO);
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 8) {
    // ================= TMA producer =================
    if (lane == 0) {
      const uint64_t pol_kv = policy_evict_last();  // K/V are re-read by the head's other CTAs
      mbar_arrive_expect_tx(bar_q_full, ntiles * C::kTileBytes);
      for (int t = 0; t < ntiles; ++t)
        for (int a = 0; a < C::kAtoms; ++a)
          tma_load_3d(sQ + t * C::kTileBytes + a * kAtomBytes, &tmQ, bar_q_full, a * 64,
                      (2 * pr + t) * kBM, bh);
      int issued_until = 0;  // blocks [0, issued_until) were issued
      const int skip_block = debug_skip_load > 0 ? debug_skip_load / 2 : -1;  // test hook
      bool ok = true;
      for (int j = 0; j < Tmax && ok; ++j) {
        const int slot = j % C::kStages;
        const int use = j / C::kStages;
        if (use > 0) {
          ok = mbar_wait(bar_kv_empty(slot), (use - 1) & 1, abort_flag, err, kSiteKvEmpty, j);
          if (!ok) break;
        }
        if (j == skip_block) continue;
        // K_j and V_j land on one barrier
        const uint32_t dst = sRing + slot * C::kStageBytes;
        mbar_arrive_expect_tx(bar_kv_full(slot), C::kStageBytes);
        for (int a = 0; a < C::kAtoms; ++a)
          tma_load_3d_hint(dst + a * kAtomBytes, &tmK, bar_kv_full(slot), a * 64, j * kBN, bh,
                           pol_kv);
        for (int a = 0; a < C::kAtoms; ++a)
          tma_load_3d_hint(dst + C::kTileBytes + a * kAtomBytes, &tmV, bar_kv_full(slot), a * 64,
                           j * kBN, bh, pol_kv);
        issued_until = j + 1;
      }
      if (!ok) {
        // Let every copy this thread started land before the CTA unwinds.
        const int first = issued_until > C::kStages ? issued_until - C::kStages : 0;
        for (int j = first; j < issued_until; ++j) {
          if (j == skip_block) continue;
          volatile int never = 0;
          mbar_wait(bar_kv_full(j % C::kStages), (j / C::kStages) & 1, &never, nullptr,
                    kSiteDrain, j);
        }
        volatile int never = 0;
        mbar_wait(bar_q_full, 0, &never, nullptr, kSiteDrain, -1);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ================= MMA issuer =================
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_bf16(kBM, kBN, false, false);
      constexpr uint32_t kIdescPV = idesc_bf16(kBM, D, false, true);
      // Base descriptors are built once; each MMA then adds a compile-time
      // offset to the 14-bit start-address field (which never carries: every
      // shared address is below 256 KB), keeping the issue loop short.
      const uint64_t qd0 = sdesc_sw128(sQ, 16, 1024);
      const uint64_t kd0 = sdesc_sw128(sRing, 16, 1024);
      const uint64_t vd0 = sdesc_sw128(sRing, kAtomBytes, 1024);
      bool ok = mbar_wait(bar_q_full, 0, abort_flag, err, kSiteQFull, 0);
      tc_fence_after();

      // S_t = Q_t K_j^T (its wait also covers V_j, which shares the stage)
      auto issue_s = [&](int t, int j) -> bool {
        const int slot = j % C::kStages;
        if (!mbar_wait(bar_kv_full(slot), (j / C::kStages) & 1, abort_flag, err, kSiteKvFull,
                       j))
          return false;
        tc_fence_after();
        const uint64_t qb = qd0 + (uint64_t)(t * (C::kTileBytes >> 4));
        const uint64_t kb = kd0 + (uint64_t)(slot * (C::kStageBytes >> 4));
        const uint32_t dS = tbase + C::kColS + t * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = (uint64_t)(((kk >> 2) * kAtomBytes + (kk & 3) * 32) >> 4);
          mma_ss(dS, qb + off, kb + off, kIdescS, kk > 0);
        }
        tc_commit(bar_s_full(t));
        return true;
      };
      // O_t += P_t V_j in two halves of 64 keys: the softmax of tile t hands
      // each half h of P_t over on p_full[t][h], and that half's MMAs are
      // committed to pv_done[t][h] (each completes once per block).
      auto issue_pv = [&](int t, int j) -> bool {
        const int slot = j % C::kStages;
        const uint64_t vb = vd0 + (uint64_t)((slot * C::kStageBytes + C::kTileBytes) >> 4);
        const uint32_t dO = tbase + C::kColO + t * 128;
        const uint32_t aP = tbase + C::kColS + t * 128;
        const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (!mbar_wait(bar_p_full(t, h), j & 1, abort_flag, err, kSitePFull, 2 * j + h))
            return false;
          tc_fence_after();
#pragma unroll
          for (int kk = 4 * h; kk < 4 * h + 4; ++kk) {
            // A = P (bf16, 2 per TMEM column): keys [16kk, 16kk+16) = 8 columns.
            // B = V block, MN-major: 16 keys = 2 groups of 8 rows of 128 B.
            mma_ts(dO, aP + kk * 8, vb + (uint64_t)((kk * 16 * 128) >> 4), kIdescPV,
                   kk > 0 ? 1u : acc0);
          }
          tc_commit(bar_pv_done(t, h));
        }
        // the stage of block j is free once the last tile reading it is done
        const int last_t = (j < Tt[1]) ? 1 : 0;
        if (t == last_t) tc_commit(bar_kv_empty(slot));
        return true;
      };

      for (int t = 0; t < kTilesPerCta && ok; ++t)
        if (Tt[t] > 0) ok = issue_s(t, 0);
      for (int j = 0; j < Tmax && ok; ++j) {
        for (int t = 0; t < kTilesPerCta && ok; ++t) {
          if (j >= Tt[t]) continue;
          ok = issue_pv(t, j);
          if (ok && j + 1 < Tt[t]) ok = issue_s(t, j + 1);
        }
      }
      // Every MMA this thread issued must be complete before TMEM is freed.
      tc_commit(bar_mma_drain);
      volatile int never = 0;
      mbar_wait(bar_mma_drain, 0, &never, nullptr, kSiteDrain, -2);
    }
    __syncwarp();
  } else {
    // ================= softmax warpgroups (tile t = warp / 4) ==============
    const int t = warp >> 2;
    const int T = Tt[t];
    const int r = threadIdx.x & 127;  // row within the Q tile == TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tbase + lane_off + C::kColS + t * 128;
    const uint32_t tO = tbase + lane_off + C::kColO + t * 128;
    const int q0 = (2 * pr + t) * kBM;
    const int row = q0 + r;
    const int lim = kCausal ? min(N, row + 1) : N;  // keys [0, lim) are visible
    float m_ref = -INFINITY;  // running max (log2 units), lazily updated
    float l = 0.f;
    bool ok = true;

    for (int j = 0; j < T; ++j) {
      ok = mbar_wait(bar_s_full(t), j & 1, abort_flag, err, kSiteSFull, j);
      ok = __all_sync(0xffffffffu, ok);  // tcgen05.ld/st below are warp-collective
      if (!ok) break;
      tc_fence_after();
      // Each 64-key half of the block is an online-softmax step of its own:
      // its P is handed to the MMA thread as soon as it is written, so the PV
      // MMAs of the first half run while the second half is computed.
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        const int nvalid = lim - j * kBN - h * 64;  // keys c < nvalid of this half are visible
        const bool full = nvalid >= 64;
        const uint32_t tSh = tS + h * 64;  // this half's 64 S columns
        const uint32_t tPh = tS + h * 32;  // its P (bf16 pairs, over already-read S columns)
        float alpha = 1.f;
        bool resc = false;
        uint32_t p[32];
        // Fast path (reference set, scale >= 0): P = 2^(scale*s - m_ref) with
        // the CURRENT reference and no row max.  It is kept when every row
        // sum of the half is at most kFastSumLimit, which bounds every P by
        // that limit; otherwise S, still intact in TMEM, is reloaded and the
        // half takes the slow path with its exact max.
        bool done = false;
        if (__all_sync(0xffffffffu, m_ref != -INFINITY && scale_log2 >= 0.f)) {
          float sh[64], rr[8];
          const float nm = -m_ref;
#pragma unroll
          for (int u = 0; u < 8; ++u) rr[u] = 0.f;
          tmem_ld64(tSh, sh);
          // a half crossing the causal diagonal or the end of the keys gives
          // its invisible keys P = 0 (the row-sum bound holds all the same)
          if (__all_sync(0xffffffffu, full)) {
#pragma unroll
            for (int c = 0; c < 64; c += 8) {
              float tv[8], pv[8];
#pragma unroll
              for (int u = 0; u < 8; u += 2)
                ffma2(tv[u], tv[u + 1], sh[c + u], sh[c + u + 1], scale_log2, scale_log2, nm, nm);
#pragma unroll
              for (int u = 0; u < 8; ++u) pv[u] = fast_exp2(tv[u]);
#pragma unroll
              for (int u = 0; u < 8; u += 2) fadd2_acc(rr[u], rr[u + 1], pv[u], pv[u + 1]);
#pragma unroll
              for (int u = 0; u < 8; u += 2) p[(c + u) / 2] = pack_bf16x2(pv[u], pv[u + 1]);
            }
          } else {
#pragma unroll
            for (int c = 0; c < 64; c += 8) {
              float tv[8], pv[8];
#pragma unroll
              for (int u = 0; u < 8; u += 2)
                ffma2(tv[u], tv[u + 1], sh[c + u], sh[c + u + 1], scale_log2, scale_log2, nm, nm);
#pragma unroll
              for (int u = 0; u < 8; ++u) pv[u] = (c + u < nvalid) ? fast_exp2(tv[u]) : 0.f;
#pragma unroll
              for (int u = 0; u < 8; u += 2) fadd2_acc(rr[u], rr[u + 1], pv[u], pv[u + 1]);
#pragma unroll
              for (int u = 0; u < 8; u += 2) p[(c + u) / 2] = pack_bf16x2(pv[u], pv[u + 1]);
            }
          }
          const float rs = ((rr[0] + rr[1]) + (rr[2] + rr[3])) + ((rr[4] + rr[5]) + (rr[6] + rr[7]));
          if (__all_sync(0xffffffffu, rs <= kFastSumLimit)) {
            tmem_st32(tPh, p);
            l += rs;
            done = true;
          }
        }
        if (!done) {
          float sv[64];
          tmem_ld64(tSh, sv);  // S of this half is intact (no P stored over it yet)
          float mt;
          if (full) {
            // max of scale*s is scale*max(s) (or scale*min(s) for a negative scale)
            float a0 = sv[0], a1 = sv[1], a2 = sv[2], a3 = sv[3];
            if (scale_log2 >= 0.f) {
#pragma unroll
              for (int c = 4; c < 64; c += 4) {
                a0 = fmaxf(a0, sv[c]); a1 = fmaxf(a1, sv[c + 1]);
                a2 = fmaxf(a2, sv[c + 2]); a3 = fmaxf(a3, sv[c + 3]);
              }
              mt = fmaxf(fmaxf(a0, a1), fmaxf(a2, a3)) * scale_log2;
            } else {
#pragma unroll
              for (int c = 4; c < 64; c += 4) {
                a0 = fminf(a0, sv[c]); a1 = fminf(a1, sv[c + 1]);
                a2 = fminf(a2, sv[c + 2]); a3 = fminf(a3, sv[c + 3]);
              }
              mt = fminf(fminf(a0, a1), fminf(a2, a3)) * scale_log2;
            }
          } else {
            mt = -INFINITY;
#pragma unroll
            for (int c = 0; c < 64; ++c) {
              sv[c] = (c < nvalid) ? sv[c] * scale_log2 : -INFINITY;
              mt = fmaxf(mt, sv[c]);
            }
          }
          const float m_new = fmaxf(m_ref, mt);
          resc = m_new > m_ref + kRescaleThreshold;  // false while both -inf
          if (resc) {
            alpha = fast_exp2(m_ref - m_new);  // 0 when m_ref == -inf
            m_ref = m_new;
            l *= alpha;
          }
          const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
          float r0 = 0.f, r1 = 0.f, r2 = 0.f, r3 = 0.f;
#pragma unroll
          for (int c = 0; c < 64; c += 4) {
            float p0, p1, p2, p3;
            if (full) {
              p0 = fast_exp2(fmaf(sv[c], scale_log2, -m_use));
              p1 = fast_exp2(fmaf(sv[c + 1], scale_log2, -m_use));
              p2 = fast_exp2(fmaf(sv[c + 2], scale_log2, -m_use));
              p3 = fast_exp2(fmaf(sv[c + 3], scale_log2, -m_use));
            } else {
              p0 = fast_exp2(sv[c] - m_use);
              p1 = fast_exp2(sv[c + 1] - m_use);
              p2 = fast_exp2(sv[c + 2] - m_use);
              p3 = fast_exp2(sv[c + 3] - m_use);
            }
            r0 += p0; r1 += p1; r2 += p2; r3 += p3;
            p[c / 2] = pack_bf16x2(p0, p1);
            p[c / 2 + 1] = pack_bf16x2(p2, p3);
          }
          tmem_st32(tPh, p);
          l += (r0 + r1) + (r2 + r3);
        }

        // Lazy correction of O before this half's PV: needed only if some row
        // of this warp moved its reference, and only once every earlier PV of
        // the tile has landed: the second half of block j-1 (h = 0) or the
        // first half of block j (h = 1).
        if ((j > 0 || h > 0) && __any_sync(0xffffffffu, resc)) {
          ok = h == 0 ? mbar_wait(bar_pv_done(t, 1), (j - 1) & 1, abort_flag, err, kSitePvDone,
                                  2 * j)
                      : mbar_wait(bar_pv_done(t, 0), j & 1, abort_flag, err, kSitePvDone,
                                  2 * j + 1);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            float ov[32];
            tmem_ld32(tO + c * 32, ov);
            uint32_t ou[32];
#pragma unroll
            for (int u = 0; u < 32; ++u) ou[u] = __float_as_uint(ov[u] * alpha);
            tmem_st32(tO + c * 32, ou);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar_p_full(t, h));
      }
      if (!ok) break;
    }

    if (T > 0) {
      if (ok) ok = mbar_wait(bar_pv_done(t, 1), (T - 1) & 1, abort_flag, err, kSitePvDone, 2 * T);
      ok = __all_sync(0xffffffffu, ok);
      const uint32_t stage_addr = sQ + t * C::kTileBytes;  // Q_t is no longer read
      if (ok) {
        tc_fence_after();
        // ---- epilogue: O / l -> bf16 into the Q_t buffer, then TMA store
        const float inv_l = 1.0f / l;
        uint8_t* stage = smem + C::kQOff + t * C::kTileBytes;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          float ov[32];
          tmem_ld32(tO + c * 32, ov);
          const int atom = (c * 32) / 64;
          const int chunk0 = ((c * 32) % 64) / 8;  // 16-byte chunk within the 128-B row
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 w;
            w.x = pack_bf16x2(ov[q4 * 8 + 0] * inv_l, ov[q4 * 8 + 1] * inv_l);
            w.y = pack_bf16x2(ov[q4 * 8 + 2] * inv_l, ov[q4 * 8 + 3] * inv_l);
            w.z = pack_bf16x2(ov[q4 * 8 + 4] * inv_l, ov[q4 * 8 + 5] * inv_l);
            w.w = pack_bf16x2(ov[q4 * 8 + 6] * inv_l, ov[q4 * 8 + 7] * inv_l);
            const int phys = (chunk0 + q4) ^ (r & 7);  // 128-byte swizzle
            *reinterpret_cast<uint4*>(stage + atom * kAtomBytes + r * 128 + phys * 16) = w;
          }
        }
        fence_proxy_async_smem();
        if (row < N) {
          constexpr float kLn2 = 0.69314718055994530942f;
          lse[(size_t)bh * N + row] = (m_ref + log2f(l)) * kLn2;
        }
      }
      // All four warps of this warpgroup reach this barrier on every path
      // (their waits are bounded); the store is skipped if any role aborted.
      named_barrier_sync(1 + t, 128);
      if (r == 0 && *abort_flag == 0) {
        for (int a = 0; a < C::kAtoms; ++a)
          tma_store_3d(&tmO, stage_addr + a * kAtomBytes, a * 64, q0, bh);
        bulk_commit();
        bulk_wait_all();
      }
    }
  }

  // ---- teardown: every role has finished (or unwound); free TMEM
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tbase, C::kTmemCols);
  }
}

CUresult make_map_3d(CUtensorMap* map, const void* ptr, int D, int N, int BH) {
  PFN_encodeTiled enc = get_encode_tiled();
  if (!enc) return CUDA_ERROR_NOT_FOUND;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)N * D * 2};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

long long num_ctas(int B, int H, int N) {
  const int n_qt = (N + kBM - 1) / kBM;
  return (long long)((n_qt + 1) / 2) * B * H;
}

template <int D, bool kCausal>
cudaError_t launch_t(const PrefillBf16Args& a, const CUtensorMap& mq, const CUtensorMap& mk,
                     const CUtensorMap& mv, const CUtensorMap& mo, cudaStream_t s) {
  using C = Cfg<D>;
  auto kern = prefill_bf16_kernel<D, kCausal>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const float scale_log2 = a.scale * 1.4426950408889634f;
  kern<<<(unsigned)num_ctas(a.B, a.H, a.N), kThreads, C::kSmemBytes, s>>>(
      mq, mk, mv, mo, a.lse, a.B * a.H, a.N, scale_log2, a.err, a.debug_skip_load);
  return cudaGetLastError();
}

}  // namespace

bool prefill_bf16_info(int D, int* Br, int* Bc, int* threads, int* smem) {
  int bytes;
  if (D == 128) bytes = Cfg<128>::kSmemBytes;
  else if (D == 64) bytes = Cfg<64>::kSmemBytes;
  else return false;
  if (Br) *Br = kBM;
  if (Bc) *Bc = kBN;
  if (threads) *threads = kThreads;
  if (smem) *smem = bytes;
  return true;
}

cudaError_t launch_prefill_bf16(const PrefillBf16Args& a, cudaStream_t s) {
  const long long blocks = num_ctas(a.B, a.H, a.N);
  if (blocks > 0x7fffffffLL) {
    attn_set_error("attn_fwd: too many query blocks (%lld)", blocks);
    return cudaErrorInvalidValue;
  }
  const int BH = a.B * a.H;
  CUtensorMap mq, mk, mv, mo;
  CUresult r = make_map_3d(&mq, a.q, a.D, a.N, BH);
  if (r == CUDA_SUCCESS) r = make_map_3d(&mk, a.k, a.D, a.N, BH);
  if (r == CUDA_SUCCESS) r = make_map_3d(&mv, a.v, a.D, a.N, BH);
  if (r == CUDA_SUCCESS) r = make_map_3d(&mo, a.o, a.D, a.N, BH);
  if (r != CUDA_SUCCESS) {
    attn_set_error("attn_fwd: cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return cudaErrorInvalidValue;
  }
  if (a.D == 128)
    return a.causal ? launch_t<128, true>(a, mq, mk, mv, mo, s)
                    : launch_t<128, false>(a, mq, mk, mv, mo, s);
  return a.causal ? launch_t<64, true>(a, mq, mk, mv, mo, s)
                  : launch_t<64, false>(a, mq, mk, mv, mo, s);
}
