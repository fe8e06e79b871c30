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
// Hopper or RTX kernels).  A work item is TWO consecutive 128-row Q tiles of
// one head, whose K/V blocks are streamed once for both.  The kernel is
// persistent (one CTA per SM); each CTA runs items one after another:
//   * warp 8  : TMA producer and work source.  Per item: each Q tile as soon
//               as the previous item's last S MMA of that tile is done, then
//               K_j and V_j together into a ring of stages (128-byte
//               swizzle), one full and one empty mbarrier per stage; with the
//               causal mask also K/V block j+1 into L2 right after block j's
//               load.  The next item is claimed from the launch's ticket
//               counter five blocks before this one's last load, so items
//               go to the CTAs that free up first (in a causal item its Q_0
//               goes out right after tile 0's last block); its number reaches
//               the other warps through a 4-slot ring in shared memory.
//   * warp 9  : MMA issuer (one thread) and TMEM owner.  For tile t,
//               S_t = Q_t K_j^T (tcgen05.mma M=128 N=128 K=D) into TMEM, and
//               O_t += P_t V_j with P read straight from TMEM as the A operand,
//               in two halves of 64 keys.  The issue order S0_0, S1_0, PV0_0,
//               S0_1, PV1_0, S1_1, ... lets the tensor core work on one tile
//               while the other tile's softmax runs (ping-pong).  Per-block
//               barrier phases run on across items.
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
//               rescale; exact because O and l share the stale reference).
//               The epilogue reads O_t out of TMEM (releasing it to the next
//               item's first PV), then O/l -> bf16 one 64-column atom at a time
//               through the tile's own 16 KB staging buffer -> TMA store, LSE.
//   TMEM columns: S0 [0,128), S1 [128,256), O0 [256,384), O1 [384,512).
//   Item order: heads in groups of 16 (causal) or 8 (no mask), so that the
//   CTAs running together share those heads' K/V in L2; heaviest causal Q
//   pairs first within a group.
//   Every wait is bounded (about 2 s); a stuck pipeline records
//   ATTN_ERR_DEVICE_TIMEOUT and the CTA unwinds, frees TMEM and exits.
#include <math.h>

#include <atomic>
#include <mutex>
#include <type_traits>

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
// heads scheduled together: 16 for causal, 8 without a mask (measured best of
// 8 / 16 / 32 / 64 on B4 H16 N4096 D128 for each)
template <bool kCausal>
constexpr int kHeadGroup = kCausal ? 16 : 8;
constexpr int kItemSlots = 4;              // work items handed from the producer to the others

template <int D>
struct Cfg {
  static constexpr int kAtoms = D / 64;
  static constexpr int kTileBytes = kAtoms * kAtomBytes;  // Q, K or V block
  static constexpr int kStageBytes = 2 * kTileBytes;      // K_j then V_j
  static constexpr int kStages = (D == 128) ? 2 : 5;      // ring slots (one KV block each)
  static constexpr int kQOff = 0;                          // Q0, Q1
  static constexpr int kRingOff = kTilesPerCta * kTileBytes;
  static constexpr int kOutOff = kRingOff + kStages * kStageBytes;  // O staging, one atom per tile
  static constexpr int kBarOff = kOutOff + kTilesPerCta * kAtomBytes;
  // barriers: q_full[tile], q_free[tile], kv_full[S], kv_empty[S], s_full[tile],
  // p_full[tile] (+1 unused), pv_done[tile] (+1 unused), o_free[tile],
  // item_full[4], item_empty[4], mma_drain.  p_full[t] completes once per KV
  // block and pv_done[t] once per item, so no waiter is ever two phases
  // behind or ahead of one.
  static constexpr int kNumBars = 2 + 2 + 2 * kStages + 2 + 4 + 4 + 2 + 2 * kItemSlots + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // tmem base, abort flag, item ring
  static constexpr int kSmemBytes = kMiscOff + 32 + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;    // + 128 * tile
  static constexpr uint32_t kColO = 256;  // + 128 * tile
};

// A work item is a pair of consecutive Q tiles of one head.  Items are
// numbered in heads of groups of kHeadGroup<kCausal> (the CTAs running together share
// those heads' K/V in L2) and, within a group, heaviest causal pairs first.
struct Item {
  int bh, pr;
  int T[kTilesPerCta];  // KV blocks visited by each Q tile (0: tile absent)
};

template <bool kCausal>
__device__ __forceinline__ Item decode_item(int item, int BH, int N) {
  const int n_qt = (N + kBM - 1) / kBM;
  const int n_pairs = (n_qt + 1) / 2;
  constexpr int HG = kHeadGroup<kCausal>;
  const int group = item / (HG * n_pairs);
  const int g_heads = min(HG, BH - group * HG);
  const int rem = item - group * HG * n_pairs;
  Item it;
  it.bh = group * HG + rem % g_heads;
  it.pr = kCausal ? (n_pairs - 1 - rem / g_heads) : (rem / g_heads);
#pragma unroll
  for (int t = 0; t < kTilesPerCta; ++t) {
    const int qt = 2 * it.pr + t;
    if (qt >= n_qt) {
      it.T[t] = 0;
    } else {
      const int kv_limit = kCausal ? min(qt * kBM + kBM, N) : N;
      it.T[t] = (kv_limit + kBN - 1) / kBN;
    }
  }
  return it;
}

template <int D, bool kCausal>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_bf16_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV,
                        const __grid_constant__ CUtensorMap tmO, float* __restrict__ lse,
                        int BH, int N, float scale_log2, int* err, int* ticket, int debug_skip_load) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment: swizzle atoms must start on a 1024-byte boundary.
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);

  const uint32_t sQ = base + C::kQOff;
  const uint32_t sRing = base + C::kRingOff;
  const uint32_t bar0 = base + C::kBarOff;
  auto bar_q_full = [&](int t) { return bar0 + 8u * t; };
  auto bar_q_free = [&](int t) { return bar0 + 8u * (2 + t); };
  auto bar_kv_full = [&](int s) { return bar0 + 8u * (4 + s); };
  auto bar_kv_empty = [&](int s) { return bar0 + 8u * (4 + C::kStages + s); };
  auto bar_s_full = [&](int t) { return bar0 + 8u * (4 + 2 * C::kStages + t); };
  auto bar_p_full = [&](int t) { return bar0 + 8u * (6 + 2 * C::kStages + t); };
  auto bar_pv_done = [&](int t) { return bar0 + 8u * (10 + 2 * C::kStages + t); };
  auto bar_o_free = [&](int t) { return bar0 + 8u * (14 + 2 * C::kStages + t); };
  auto bar_item_full = [&](int i) { return bar0 + 8u * (16 + 2 * C::kStages + i); };
  auto bar_item_empty = [&](int i) {
    return bar0 + 8u * (16 + 2 * C::kStages + kItemSlots + i);
  };
  const uint32_t bar_mma_drain = bar0 + 8u * (16 + 2 * C::kStages + 2 * kItemSlots);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 4);
  volatile int* item_ring = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 16);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_qt = (N + kBM - 1) / kBM;
  const int total_items = ((n_qt + 1) / 2) * BH;

  // ---- setup: barriers (thread 0), TMEM (warp 9)
  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar_q_full(t), 1);
      mbar_init(bar_q_free(t), 1);
      mbar_init(bar_s_full(t), 1);
      mbar_init(bar_o_free(t), 128);
      mbar_init(bar_p_full(t), 128);
      mbar_init(bar_pv_done(t), 1);
    }
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar_kv_full(s), 1);
      mbar_init(bar_kv_empty(s), 1);
    }
    for (int i = 0; i < kItemSlots; ++i) {
      mbar_init(bar_item_full(i), 1);
      mbar_init(bar_item_empty(i), 1 + 256);  // the MMA thread and every softmax thread
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
    // ================= TMA producer and work-item source =================
    if (lane == 0) {
      const uint64_t pol_kv = policy_evict_last();  // K/V are re-read by the head's other CTAs
      const int skip_block = debug_skip_load > 0 ? debug_skip_load / 2 : -1;  // test hook
      int kv = 0;             // K/V blocks this CTA has loaded (ring position)
      uint32_t skipped = 0;   // bit (kv % 32): that load was skipped by the test hook
      int qn[2] = {0, 0};     // Q loads per tile
      bool ok = true;
      int item = blockIdx.x;  // first item; later ones come from the launch's ticket
      bool q0_issued = false; // this item's Q_0 went out during the previous item
      for (int k = 0; ok; ++k) {
        const int slot = k % kItemSlots;
        if (k >= kItemSlots) {
          ok = mbar_wait(bar_item_empty(slot), (k / kItemSlots - 1) & 1, abort_flag, err,
                         kSiteQFull, k);
          if (!ok) break;
        }
        item_ring[slot] = item < total_items ? item : -1;
        mbar_arrive(bar_item_full(slot));
        if (item >= total_items) break;
        const Item it = decode_item<kCausal>(item, BH, N);
        // Q_t of this item once the previous item's last S of that tile is
        // done.  Q_0 goes first, then K/V block 0, then Q_1: tile 1 runs one
        // block longer than tile 0 at the end of a causal item, and block 0
        // need not wait for that.
        auto load_q = [&](const Item& iq, int t) -> bool {
          if (iq.T[t] == 0) return true;
          if (qn[t] > 0 &&
              !mbar_wait(bar_q_free(t), (qn[t] - 1) & 1, abort_flag, err, kSiteQFull, k))
            return false;
          mbar_arrive_expect_tx(bar_q_full(t), C::kTileBytes);
          for (int a = 0; a < C::kAtoms; ++a)
            tma_load_3d(sQ + t * C::kTileBytes + a * kAtomBytes, &tmQ, bar_q_full(t), a * 64,
                        (2 * iq.pr + t) * kBM, iq.bh);
          ++qn[t];
          return true;
        };
        if (!q0_issued) ok = load_q(it, 0);
        q0_issued = false;
        if (!ok) break;
        const int Tmax = max(it.T[0], it.T[1]);
        // The next item is claimed five blocks before this item's last K/V
        // load, so that the claim's round trip to the counter (1-2.5 us) is
        // hidden behind those loads (three, five, six and eight measured;
        // five on); items still go to the CTAs that free up first.
        // When tile 1 runs a block longer (causal), the next item's Q_0 goes
        // out right after tile 0's last K/V block: its buffer is free once
        // tile 0's last S is done, which comes before tile 1's last block is
        // loaded, so it is no longer late when the next item starts (issuing
        // that item's first S ahead of tile 1's last PV, or an L2 prefetch of
        // its Q tiles, measured slower).
        const int j_claim = max(0, Tmax - 5);
        const bool early_q0 = kCausal && it.T[1] == it.T[0] + 1;
        int next = total_items;
        for (int j = 0; j < Tmax; ++j, ++kv) {
          if (j == j_claim) next = (int)gridDim.x + atomicAdd(ticket, 1);
          const int s = kv % C::kStages;
          const int use = kv / C::kStages;
          if (use > 0) {
            ok = mbar_wait(bar_kv_empty(s), (use - 1) & 1, abort_flag, err, kSiteKvEmpty, j);
            if (!ok) break;
          }
          if (j == skip_block) {
            skipped |= 1u << (kv & 31);
          } else {
            skipped &= ~(1u << (kv & 31));
            // K_j and V_j land on one barrier
            const uint32_t dst = sRing + s * C::kStageBytes;
            mbar_arrive_expect_tx(bar_kv_full(s), C::kStageBytes);
            for (int a = 0; a < C::kAtoms; ++a)
              tma_load_3d_hint(dst + a * kAtomBytes, &tmK, bar_kv_full(s), a * 64, j * kBN,
                               it.bh, pol_kv);
            for (int a = 0; a < C::kAtoms; ++a)
              tma_load_3d_hint(dst + C::kTileBytes + a * kAtomBytes, &tmV, bar_kv_full(s), a * 64,
                               j * kBN, it.bh, pol_kv);
          }
          // causal: block j+1 into L2 now, so that its load (issued once a
          // stage frees) is served from L2 (one block ahead measured best of
          // one to three; without a mask the prefetch costs more than it
          // saves).  Where the next item's Q_0 goes out at this block, the
          // prefetch follows it, so that the Q tile, whose arrival sets the
          // item boundary, does not queue behind it.
          auto prefetch_next_block = [&]() {
            if (kCausal && j + 1 < Tmax)
              for (int a = 0; a < C::kAtoms; ++a) {
                tma_prefetch_3d(&tmK, a * 64, (j + 1) * kBN, it.bh);
                tma_prefetch_3d(&tmV, a * 64, (j + 1) * kBN, it.bh);
              }
          };
          const bool q0_here = early_q0 && j == it.T[0] - 1 && next < total_items;
          if (!q0_here) prefetch_next_block();
          if (j == 0) {
            ok = load_q(it, 1);
            if (!ok) break;
          }
          if (q0_here) {
            ok = load_q(decode_item<kCausal>(next, BH, N), 0);
            if (!ok) break;
            q0_issued = true;
            prefetch_next_block();
          }
        }
        item = next;
      }
      if (!ok) {
        // Let every copy this thread started land before the CTA unwinds.
        const int first = kv > C::kStages ? kv - C::kStages : 0;
        for (int x = first; x < kv; ++x) {
          if (skipped & (1u << (x & 31))) continue;
          volatile int never = 0;
          mbar_wait(bar_kv_full(x % C::kStages), (x / C::kStages) & 1, &never, nullptr,
                    kSiteDrain, x);
        }
        for (int t = 0; t < kTilesPerCta; ++t) {
          if (qn[t] == 0) continue;
          volatile int never = 0;
          mbar_wait(bar_q_full(t), (qn[t] - 1) & 1, &never, nullptr, kSiteDrain, -1);
        }
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
      int kv = 0;                // ring position of the current item's block 0
      int bc0 = 0, bc1 = 0;      // KV blocks each tile has been through (barrier phases)
      int qn0 = 0, qn1 = 0;      // items each tile has been loaded for
      int T0 = 0, T1 = 0;        // the current item's KV blocks per tile
      int pb0 = 0, pb1 = 0;      // phase offsets of the tiles' per-block barriers
      bool ok = true;
      using Tile0 = std::integral_constant<int, 0>;
      using Tile1 = std::integral_constant<int, 1>;

      // S_t = Q_t K_j^T (its wait also covers V_j, which shares the stage).
      // The tile is a compile-time constant so that the issue path carries
      // no per-tile selects: every instruction of this thread delays the pipe.
      // Where the other tile's S of the same block was issued just before
      // (tile 1's S of any block that tile 0 also visits), the stage is known
      // to be full and the wait is left out.
      using Wait = std::true_type;
      using NoWait = std::false_type;
      auto issue_s = [&](auto tile, int j, auto wait) -> bool {
        constexpr int t = decltype(tile)::value;
        const int x = kv + j;
        const int slot = x % C::kStages;
        if constexpr (decltype(wait)::value) {
          if (!mbar_wait(bar_kv_full(slot), (x / C::kStages) & 1, abort_flag, err, kSiteKvFull,
                         j))
            return false;
          tc_fence_after();
        }
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
      // O_t += P_t V_j: the softmax of tile t hands the block's P over on
      // p_full[t].  pv_done[t] is committed only after the tile's last block
      // of an item, for the epilogue: within an item the next block's S
      // commit already covers this PV (a commit tracks every earlier MMA of
      // this thread).  The steady loop, which never holds a last block,
      // passes NotLast and skips the test.
      using MaybeLast = std::true_type;
      using NotLast = std::false_type;
      auto issue_pv = [&](auto tile, int j, auto may_be_last) -> bool {
        constexpr int t = decltype(tile)::value;
        const int x = kv + j;
        const int slot = x % C::kStages;
        const int ph = (j & 1) ^ (t ? pb1 : pb0);
        const uint64_t vb = vd0 + (uint64_t)((slot * C::kStageBytes + C::kTileBytes) >> 4);
        const uint32_t dO = tbase + C::kColO + t * 128;
        const uint32_t aP = tbase + C::kColS + t * 128;
        const uint32_t acc0 = j > 0 ? 1u : 0u;
        if (!mbar_wait(bar_p_full(t), ph, abort_flag, err, kSitePFull, j)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          // A = P (bf16, 2 per TMEM column): keys [16kk, 16kk+16) = 8 columns.
          // B = V block, MN-major: 16 keys = 2 groups of 8 rows of 128 B.
          mma_ts(dO, aP + kk * 8, vb + (uint64_t)((kk * 16 * 128) >> 4), kIdescPV,
                 kk > 0 ? 1u : acc0);
        }
        if constexpr (decltype(may_be_last)::value) {
          if (j == (t ? T1 : T0) - 1) tc_commit(bar_pv_done(t));
        }
        // the stage of block j is free once the last tile reading it is done
        if (t == 1 || j >= T1) tc_commit(bar_kv_empty(slot));
        return true;
      };
      // the first PV of tile t in an item overwrites O_t: the previous
      // item's epilogue must have read it
      auto wait_o_free = [&](auto tile) -> bool {
        constexpr int t = decltype(tile)::value;
        const int qn = t ? qn1 : qn0;
        if (qn == 0) return true;
        if (!mbar_wait(bar_o_free(t), (qn - 1) & 1, abort_flag, err, kSitePvDone, qn))
          return false;
        tc_fence_after();
        return true;
      };

      for (int k = 0; ok; ++k) {
        const int islot = k % kItemSlots;
        ok = mbar_wait(bar_item_full(islot), (k / kItemSlots) & 1, abort_flag, err, kSiteQFull, k);
        if (!ok) break;
        const int item = item_ring[islot];
        mbar_arrive(bar_item_empty(islot));
        if (item < 0) break;
        const Item it = decode_item<kCausal>(item, BH, N);
        T0 = it.T[0];  // tile 0 is always present
        T1 = it.T[1];
        pb0 = bc0 & 1;
        pb1 = bc1 & 1;
        const int Tmax = max(T0, T1);
        // block 0 of both tiles (Q waits, O hand-over from the last item)
        ok = mbar_wait(bar_q_full(0), qn0 & 1, abort_flag, err, kSiteQFull, k);
        if (ok) {
          tc_fence_after();
          ok = issue_s(Tile0{}, 0, Wait{});
        }
        if (ok && T1 > 0) {
          ok = mbar_wait(bar_q_full(1), qn1 & 1, abort_flag, err, kSiteQFull, k);
          if (ok) {
            tc_fence_after();
            ok = issue_s(Tile1{}, 0, NoWait{});  // tile 0's S of block 0 waited
          }
        }
        // q_free[t] is committed right after the tile's last S: the producer
        // then loads the next item's Q_t while this item's tail still runs.
        if (ok && T0 == 1) tc_commit(bar_q_free(0));
        if (ok && T1 == 1) tc_commit(bar_q_free(1));
        if (ok) ok = wait_o_free(Tile0{}) && issue_pv(Tile0{}, 0, MaybeLast{});
        if (ok && T0 > 1) {
          ok = issue_s(Tile0{}, 1, Wait{});
          if (ok && T0 == 2) tc_commit(bar_q_free(0));
        }
        if (ok && T1 > 0) ok = wait_o_free(Tile1{}) && issue_pv(Tile1{}, 0, MaybeLast{});
        if (ok && T1 > 1) {
          ok = T0 > 1 ? issue_s(Tile1{}, 1, NoWait{}) : issue_s(Tile1{}, 1, Wait{});
          if (ok && T1 == 2) tc_commit(bar_q_free(1));
        }
        // blocks 1.. : the steady part has no last S of either tile and so
        // no conditions; the tail (at most three blocks) has them.
        const int Tmin = T1 > 0 ? min(T0, T1) : T0;
        const int j_tail = max(1, Tmin - 2);
        int j = 1;
        if (T1 > 0) {
          for (; j < j_tail && ok; ++j) {
            ok = issue_pv(Tile0{}, j, NotLast{});
            if (ok) ok = issue_s(Tile0{}, j + 1, Wait{});
            if (ok) ok = issue_pv(Tile1{}, j, NotLast{});
            if (ok) ok = issue_s(Tile1{}, j + 1, NoWait{});
          }
        }
        for (; j < Tmax && ok; ++j) {
          if (j < T0) {
            ok = issue_pv(Tile0{}, j, MaybeLast{});
            if (ok && j + 1 < T0) {
              ok = issue_s(Tile0{}, j + 1, Wait{});
              if (ok && j + 2 == T0) tc_commit(bar_q_free(0));
            }
          }
          if (ok && j < T1) {
            ok = issue_pv(Tile1{}, j, MaybeLast{});
            if (ok && j + 1 < T1) {
              ok = j + 1 < T0 ? issue_s(Tile1{}, j + 1, NoWait{})
                              : issue_s(Tile1{}, j + 1, Wait{});
              if (ok && j + 2 == T1) tc_commit(bar_q_free(1));
            }
          }
        }
        kv += Tmax;
        bc0 += T0;
        bc1 += T1;
        qn0 += 1;
        qn1 += T1 > 0 ? 1 : 0;
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
    const int r = threadIdx.x & 127;  // row within the Q tile == TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tbase + lane_off + C::kColS + t * 128;
    const uint32_t tO = tbase + lane_off + C::kColO + t * 128;
    const uint32_t stage_addr = base + C::kOutOff + t * kAtomBytes;  // this tile's O staging
    uint8_t* stage = smem + C::kOutOff + t * kAtomBytes;
    int bc = 0;   // KV blocks this tile has been through (barrier phases)
    int nit = 0;  // items this tile has been through (pv_done[t][1] phases)

    for (int k = 0;; ++k) {
      const int islot = k % kItemSlots;
      bool got = mbar_wait(bar_item_full(islot), (k / kItemSlots) & 1, abort_flag, err,
                           kSiteQFull, k);
      got = __all_sync(0xffffffffu, got);
      const int item = got ? item_ring[islot] : -1;
      if (got) mbar_arrive(bar_item_empty(islot));
      // the four warps take the item (or stop) together
      if (named_barrier_any(1 + t, 128, item < 0)) break;
      const Item it = decode_item<kCausal>(item, BH, N);
      const int T = t ? it.T[1] : it.T[0];
      if (T == 0) continue;
      const int bh = it.bh;
      const int q0 = (2 * it.pr + t) * kBM;
      const int row = q0 + r;
      const int lim = kCausal ? min(N, row + 1) : N;  // keys [0, lim) are visible
      float m_ref = -INFINITY;  // running max (log2 units), lazily updated
      float l = 0.f;
      bool ok = true;

      for (int j = 0; j < T; ++j) {
        ok = mbar_wait(bar_s_full(t), (bc + j) & 1, abort_flag, err, kSiteSFull, j);
        ok = __all_sync(0xffffffffu, ok);  // tcgen05.ld/st below are warp-collective
        if (!ok) break;
        tc_fence_after();
        // Each 64-key half of the block is an online-softmax step of its own
        // (its own fast-path bound and, if needed, exact max); the block's P is
        // handed to the MMA thread once, after both halves, which keeps the
        // MMA thread's waits and commits to one each per tile and block.
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

          // Lazy correction when some row of this warp moved its reference:
          // O holds every PV up to block j-1, already complete when s_full of
          // block j was seen (S_t(j) was issued after it, and a commit covers
          // every earlier MMA), so it is rescaled without a wait; and in the
          // second half the first half's P, written but not yet handed over,
          // is rescaled in TMEM too (one more bf16 rounding, on this rare path).
          if (__any_sync(0xffffffffu, resc)) {
            if (j > 0) {
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
            if (h == 1) {
              tmem_st_wait();  // the first half's P is in place before it is read back
              uint32_t pw[32];
              tmem_ld32(tS, reinterpret_cast<float*>(pw));
#pragma unroll
              for (int u = 0; u < 32; ++u) {
                const float2 f = unpack_bf16x2(pw[u]);
                pw[u] = pack_bf16x2(f.x * alpha, f.y * alpha);
              }
              tmem_st32(tS, pw);
            }
          }
        }
        // the whole block's P goes to the MMA thread in one hand-over
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar_p_full(t));

        if (!ok) break;
      }

      // ---- epilogue: O / l -> bf16, one 64-column atom at a time through this
      // tile's staging buffer, each stored by TMA; LSE.  All four warps of the
      // warpgroup reach every barrier below on every path (their waits are
      // bounded); stores are skipped once any role has aborted.
      if (ok) ok = mbar_wait(bar_pv_done(t), nit & 1, abort_flag, err, kSitePvDone, 2 * T);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) tc_fence_after();
      const float inv_l = 1.0f / l;
#pragma unroll 1
      for (int a = 0; a < C::kAtoms; ++a) {
        // the previous store from the staging buffer has read it
        if (r == 0) bulk_wait_all_read();
        named_barrier_sync(1 + t, 128);
        if (ok) {
#pragma unroll 1
          for (int c = 0; c < 2; ++c) {
            float ov[32];
            tmem_ld32(tO + a * 64 + c * 32, ov);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              uint4 w;
              w.x = pack_bf16x2(ov[q4 * 8 + 0] * inv_l, ov[q4 * 8 + 1] * inv_l);
              w.y = pack_bf16x2(ov[q4 * 8 + 2] * inv_l, ov[q4 * 8 + 3] * inv_l);
              w.z = pack_bf16x2(ov[q4 * 8 + 4] * inv_l, ov[q4 * 8 + 5] * inv_l);
              w.w = pack_bf16x2(ov[q4 * 8 + 6] * inv_l, ov[q4 * 8 + 7] * inv_l);
              const int phys = (c * 4 + q4) ^ (r & 7);  // 128-byte swizzle
              *reinterpret_cast<uint4*>(stage + r * 128 + phys * 16) = w;
            }
          }
          if (a == C::kAtoms - 1) {
            // O_t is read: the next item's first PV of this tile may overwrite it
            tc_fence_before();
            mbar_arrive(bar_o_free(t));
          }
          fence_proxy_async_smem();
        }
        const bool stop = named_barrier_any(1 + t, 128, !ok || *abort_flag != 0);
        if (r == 0 && !stop) {
          tma_store_3d(&tmO, stage_addr, a * 64, q0, bh);
          bulk_commit();
        }
        ok = ok && !stop;
      }
      if (ok && row < N) {
        constexpr float kLn2 = 0.69314718055994530942f;
        lse[(size_t)bh * N + row] = (m_ref + log2f(l)) * kLn2;
      }
      bc += T;
      ++nit;
      // one decision for the whole warpgroup: go on to the next item or stop
      if (named_barrier_any(1 + t, 128, !ok || *abort_flag != 0)) break;
    }
    if (r == 0) bulk_wait_all();  // this tile's O stores are complete
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

long long num_items(int B, int H, int N) {
  const int n_qt = (N + kBM - 1) / kBM;
  return (long long)((n_qt + 1) / 2) * B * H;
}

// Work-item tickets: each launch takes one counter, zeroes it on its stream
// (a 4-byte cudaMemsetAsync before the kernel), and its CTAs draw items from
// it.  Ordinary launches use kRoundRobinSlots counters in turn: a slot comes
// back kRoundRobinSlots launches later, by which time a launch on the same
// stream has finished, so at most kRoundRobinSlots launches on different
// streams may be in flight at once.  A launch enqueued while its stream is
// being captured into a CUDA graph gets a slot of its own for good (the
// graph replays the memset and the kernel on that slot whenever it runs), so
// a replay never shares a counter with an ordinary launch or another
// captured one.  The two replays that could still collide are replays of two
// separate instantiations of one graph running at the same time.
constexpr int kRoundRobinSlots = 64;
constexpr int kCapturedSlots = 1984;
constexpr int kTicketSlots = kRoundRobinSlots + kCapturedSlots;
__device__ int g_prefill_tickets[kTicketSlots];
std::atomic<unsigned> g_ticket_next{0};
int g_captured_next[64] = {};
void* g_ticket_base[64] = {};
std::mutex g_ticket_mu;

cudaError_t ticket_for_launch(cudaStream_t s, int** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(s, &cap);
  if (e != cudaSuccess) return e;
  void* basep = nullptr;
  int idx = 0;
  {
    std::lock_guard<std::mutex> lk(g_ticket_mu);
    if (g_ticket_base[dev] == nullptr) {
      e = cudaGetSymbolAddress(&g_ticket_base[dev], g_prefill_tickets);
      if (e != cudaSuccess) return e;
    }
    basep = g_ticket_base[dev];
    if (cap == cudaStreamCaptureStatusActive) {
      if (g_captured_next[dev] >= kCapturedSlots) {
        attn_set_error("attn_fwd: more than %d bf16 launches captured into graphs on this device",
                       kCapturedSlots);
        return cudaErrorInvalidValue;
      }
      idx = kRoundRobinSlots + g_captured_next[dev]++;
    } else {
      idx = (int)(g_ticket_next.fetch_add(1) % kRoundRobinSlots);
    }
  }
  int* slot = static_cast<int*>(basep) + idx;
  e = cudaMemsetAsync(slot, 0, sizeof(int), s);
  if (e != cudaSuccess) return e;
  *out = slot;
  return cudaSuccess;
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
  int* ticket = nullptr;
  e = ticket_for_launch(s, &ticket);
  if (e != cudaSuccess) return e;
  // persistent: one CTA per SM (the shared memory allows no more)
  const long long items = num_items(a.B, a.H, a.N);
  const unsigned grid = (unsigned)(items < a.num_sms ? items : a.num_sms);
  kern<<<grid, kThreads, C::kSmemBytes, s>>>(mq, mk, mv, mo, a.lse, a.B * a.H, a.N, scale_log2,
                                              a.err, ticket, a.debug_skip_load);
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
  const long long blocks = num_items(a.B, a.H, a.N);
  if (blocks > 0x7fffffffLL / 2) {
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
