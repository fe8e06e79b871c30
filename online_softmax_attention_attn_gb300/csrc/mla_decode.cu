// mla_decode.cu -- MLA absorbed decode on GB300 (sm_103a): split plan,
// 2-CTA-cluster tcgen05 decode kernel, and LSE combine of split partials.
//
// What it computes ("MLA x FlashAttention-3 fusion" article, hnwysp news
// 119127): each cached token is one 576-wide bf16 row [c_kv 512 | k_rope 64];
// the absorbed query [q_nope W_UK | q_rope] makes every score one 576-deep dot
// product (the absorption identity), V is the c_kv slice of the same row, and
// nothing is decompressed to global memory.  The softmax is online with a
// deferred 1/l as in the FlashAttention-2 blog (dandandamowang
// post_1787450400, sections 1.3 and 3.3); split partials are merged with
// their log-sum-exp weights (the article's "partial reduction" stage).
//
// GB300 design (not the article's Hopper sketch):
//   * The 128 query heads are the MMA M dimension against the one shared
//     latent head (M=128, tcgen05 kind::f16, fp32 accumulators in TMEM).
//   * O = 128 heads x 512 fp32 would fill all of one SM's TMEM, so a CLUSTER
//     OF TWO CTAs shares each work item by columns: rank 0 owns latent
//     columns [0,256) plus the 64 RoPE columns, rank 1 owns [256,512).  Each
//     CTA TMA-loads only its own columns of every cached row (HBM is read
//     once), computes a partial S over them, and the two partial S tiles are
//     swapped through distributed shared memory so that both hold the full S
//     and run the identical softmax.  Each then accumulates its 256 columns
//     of O = P V in TMEM (V is the same shared-memory bytes as K).
//   * Pages of 64 tokens are consumed as two 32-token steps; the block table
//     is read on the device and bounds-checked; K/V stream through a
//     5-stage mbarrier ring filled by one producer warp.
//   * Work is the flat list of all sequences' pages cut into equal chunks,
//     one chunk per cluster (persistent).  A sequence cut by a chunk edge
//     writes fp32 partials (O_s normalised, LSE_s) that a small combine
//     kernel merges; sequences inside one chunk write bf16 O directly.
//   * Every wait is bounded; a stuck pipeline records ATTN_ERR_DEVICE_TIMEOUT.
#include <math.h>

#include <mutex>

#include "common.cuh"

namespace {

using namespace gb300;

constexpr int kHq = 128;
constexpr int kDk = 576;
constexpr int kDv = 512;
constexpr int kPage = 64;
constexpr int kStep = 32;                 // tokens per pipeline step (half page)
constexpr int kThreads = 192;             // 4 softmax warps + producer + MMA
constexpr int kMaxAtoms = 5;              // 64-column atoms per CTA (rank 0)
constexpr int kQAtomBytes = kHq * 128;    // 128 heads x 64 bf16
constexpr int kKAtomBytes = kStep * 128;  // 32 tokens x 64 bf16
constexpr int kStageBytes = kMaxAtoms * kKAtomBytes;  // 20 KB
constexpr int kStages = 5;
constexpr int kXRow = 36;                 // floats per exchange row (32 + pad)
constexpr int kXBufBytes = kHq * kXRow * 4;
constexpr float kRescaleThreshold = 8.0f;

constexpr int kQOff = 0;
constexpr int kStageOff = kQOff + kMaxAtoms * kQAtomBytes;     // 80 KB
constexpr int kXOff = kStageOff + kStages * kStageBytes;        // +100 KB
constexpr int kBarOff = kXOff + 2 * kXBufBytes;                 // +36 KB
// barriers: q_full, q_empty, kv_full[S], kv_empty[S], s_full[2], xfull[2],
// xfree[2], p_full[2], pv_done, o_free, mma_drain
constexpr int kNumBars = 2 + 2 * kStages + 2 + 2 + 2 + 2 + 3;
constexpr int kMiscOff = kBarOff + kNumBars * 8;
constexpr int kSmemBytes = kMiscOff + 16 + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;     // 256 columns
constexpr uint32_t kColS = 256;   // 2 x 32 columns

// ---- workspace layout -------------------------------------------------------
struct WsLayout {
  size_t header, prefix, plse, po, total;
  int max_slots;
};

__host__ __device__ constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ constexpr WsLayout ws_layout(int B, int max_slots) {
  WsLayout w{};
  w.max_slots = max_slots;
  w.header = 0;
  w.prefix = 64;
  w.plse = align_up(w.prefix + sizeof(int) * (size_t)(B + 1), 256);
  w.po = align_up(w.plse + sizeof(float) * (size_t)max_slots * kHq, 256);
  w.total = align_up(w.po + sizeof(float) * (size_t)max_slots * kHq * kDv, 256);
  return w;
}

inline int max_chunks_for(int B, int max_blocks, int num_sms, int pps) {
  const int clusters = num_sms / 2;
  if (pps > 0) {
    const long long total = (long long)B * max_blocks;
    return (int)((total + pps - 1) / pps);
  }
  return clusters;
}

// ---- plan -------------------------------------------------------------------
// One CTA: validates lengths, writes the exclusive page prefix, the chunk
// length (pages per split) and the chunk count into the workspace header.
__global__ void __launch_bounds__(1024) mla_plan_kernel(const int32_t* __restrict__ seqlens,
                                                        int B, int max_blocks, int clusters,
                                                        int pps_override, int* __restrict__ ws_hdr,
                                                        int* __restrict__ prefix, int* err) {
  __shared__ int warp_sums[32];
  __shared__ int carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int n = 0;
    if (b < B) {
      const int L = seqlens[b];
      if (L < 0 || L > max_blocks * kPage) {
        record_error(err, ATTN_ERR_BAD_SEQLEN, 0, b);
      } else {
        n = (L + kPage - 1) / kPage;
      }
    }
    // inclusive scan within the warp, then across warps
    int x = n;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) warp_sums[wid] = x;
    __syncthreads();
    if (wid == 0) {
      int w = (lane < (int)(blockDim.x >> 5)) ? warp_sums[lane] : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, w, off);
        if (lane >= off) w += y;
      }
      warp_sums[lane] = w;
    }
    __syncthreads();
    const int incl = x + (wid > 0 ? warp_sums[wid - 1] : 0) + carry;
    if (b < B) prefix[b] = incl - n;
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) carry = incl;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const int T = carry;
    prefix[B] = T;
    int pps = pps_override > 0 ? pps_override : (T + clusters - 1) / max(clusters, 1);
    if (pps < 1) pps = 1;
    ws_hdr[0] = T;
    ws_hdr[1] = pps;
    ws_hdr[2] = (T + pps - 1) / pps;
  }
}

// ---- decode -----------------------------------------------------------------
struct Seg {
  int b, p0, p1;  // sequence and its page range [p0, p1)
  int slot;       // partial slot, or -1 when the segment is the whole sequence
};

__device__ __forceinline__ int find_batch(const int* __restrict__ prefix, int B, int page) {
  // largest b with prefix[b] <= page < prefix[b+1]
  int lo = 0, hi = B;  // search in prefix[0..B]
  while (lo < hi) {
    int mid = (lo + hi) >> 1;
    if (prefix[mid + 1] <= page) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// Enumerates the segments of chunk k in order; returns false when done.
struct ChunkIter {
  const int* prefix;
  int B, k, pps, start, end, b;
  __device__ void init(const int* pf, int B_, int k_, int pps_, int T) {
    prefix = pf; B = B_; k = k_; pps = pps_;
    start = k * pps;
    end = min(start + pps, T);
    b = (start < end) ? find_batch(prefix, B, start) : B;
  }
  __device__ bool next(Seg& s) {
    if (start >= end || b >= B) return false;
    const int seg_end = min(end, prefix[b + 1]);
    s.b = b;
    s.p0 = start - prefix[b];
    s.p1 = seg_end - prefix[b];
    const int npages = prefix[b + 1] - prefix[b];
    const bool whole = (s.p0 == 0 && s.p1 == npages);
    const bool first = (start == k * pps);
    s.slot = whole ? -1 : (first ? 2 * k : 2 * k + 1);
    start = seg_end;
    ++b;
    while (b < B && prefix[b + 1] <= start) ++b;
    return true;
  }
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tmQ,
                      const __grid_constant__ CUtensorMap tmKV,
                      const int32_t* __restrict__ block_table,
                      const int32_t* __restrict__ seqlens, __nv_bfloat16* __restrict__ o,
                      float* __restrict__ lse, const int* __restrict__ ws_hdr,
                      const int* __restrict__ prefix, float* __restrict__ part_lse,
                      float* __restrict__ part_o, int B, int max_blocks, int num_blocks,
                      float scale_log2, int* err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);

  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int cluster = blockIdx.x >> 1;
  const int nclusters = gridDim.x >> 1;
  const int T = ws_hdr[0], pps = ws_hdr[1], nchunks = ws_hdr[2];
  if (cluster >= nchunks) return;  // both CTAs of the cluster leave together

  // columns owned by this CTA, as 64-column atoms of the 576-wide row
  const int natoms = rank == 0 ? 5 : 4;
  auto atom_col = [&](int a) -> int {
    return rank == 0 ? (a < 4 ? a * 64 : 512) : (256 + a * 64);
  };

  const uint32_t sQ = base + kQOff;
  const uint32_t sStage = base + kStageOff;
  const uint32_t sX = base + kXOff;
  const uint32_t bar0 = base + kBarOff;
  const uint32_t bar_q_full = bar0, bar_q_empty = bar0 + 8;
  auto bar_kv_full = [&](int s) { return bar0 + 8u * (2 + s); };
  auto bar_kv_empty = [&](int s) { return bar0 + 8u * (2 + kStages + s); };
  auto bar_s_full = [&](int b) { return bar0 + 8u * (2 + 2 * kStages + b); };
  auto bar_xfull = [&](int b) { return bar0 + 8u * (4 + 2 * kStages + b); };
  auto bar_xfree = [&](int b) { return bar0 + 8u * (6 + 2 * kStages + b); };
  auto bar_p_full = [&](int b) { return bar0 + 8u * (8 + 2 * kStages + b); };
  const uint32_t bar_pv_done = bar0 + 8u * (10 + 2 * kStages);
  const uint32_t bar_o_free = bar0 + 8u * (11 + 2 * kStages);
  const uint32_t bar_mma_drain = bar0 + 8u * (12 + 2 * kStages);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kMiscOff + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(bar_q_full, 1);
    mbar_init(bar_q_empty, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_kv_full(s), 1);
      mbar_init(bar_kv_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_s_full(b), 1);
      mbar_init(bar_xfull(b), 128);
      mbar_init(bar_xfree(b), 128);
      mbar_init(bar_p_full(b), 128);
    }
    mbar_init(bar_pv_done, 1);
    mbar_init(bar_o_free, 128);
    mbar_init(bar_mma_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmKV);
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // peer barriers are initialised before any remote arrive
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 4) {
    // ================= producer =================
    if (lane == 0) {
      const uint64_t pol_kv = policy_evict_first();  // every cached row is read once
      int g = 0, seg_i = 0;
      int issued = 0;  // steps [0, issued) have their loads issued
      bool ok = true;
      for (int k = cluster; k < nchunks && ok; k += nclusters) {
        ChunkIter it;
        it.init(prefix, B, k, pps, T);
        Seg s;
        while (ok && it.next(s)) {
          if (seg_i > 0) {
            ok = mbar_wait(bar_q_empty, (seg_i - 1) & 1, abort_flag, err, kSiteQFull, seg_i);
            if (!ok) break;
          }
          mbar_arrive_expect_tx(bar_q_full, natoms * kQAtomBytes);
          for (int a = 0; a < natoms; ++a)
            tma_load_2d(sQ + a * kQAtomBytes, &tmQ, bar_q_full, atom_col(a), s.b * kHq);
          const int L = seqlens[s.b];
          const int t_end = min(s.p1 * kPage, L);
          for (int t = s.p0 * kPage; t < t_end && ok; t += kStep, ++g) {
            const int slot = g % kStages, use = g / kStages;
            if (use > 0) {
              ok = mbar_wait(bar_kv_empty(slot), (use - 1) & 1, abort_flag, err, kSiteKvEmpty, g);
              if (!ok) break;
            }
            int blk = block_table[(size_t)s.b * max_blocks + t / kPage];
            if (blk < 0 || blk >= num_blocks) {
              record_error(err, ATTN_ERR_BAD_BLOCK_TABLE, s.b, t / kPage);
              blk = 0;  // never read outside the pool
            }
            const int row = blk * kPage + (t % kPage);
            const uint32_t dst = sStage + slot * kStageBytes;
            mbar_arrive_expect_tx(bar_kv_full(slot), natoms * kKAtomBytes);
            for (int a = 0; a < natoms; ++a)
              tma_load_2d_hint(dst + a * kKAtomBytes, &tmKV, bar_kv_full(slot), atom_col(a), row,
                               pol_kv);
            issued = g + 1;
          }
          ++seg_i;
        }
      }
      if (!ok) {
        const int first = issued > kStages ? issued - kStages : 0;
        for (int gg = first; gg < issued; ++gg) {
          volatile int never = 0;
          mbar_wait(bar_kv_full(gg % kStages), (gg / kStages) & 1, &never, nullptr, kSiteDrain, gg);
        }
        if (seg_i > 0) {
          volatile int never = 0;
          mbar_wait(bar_q_full, (seg_i - 1) & 1, &never, nullptr, kSiteDrain, -1);
        }
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ================= MMA issuer =================
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_bf16(kHq, kStep, false, false);
      constexpr uint32_t kIdescPV = idesc_bf16(kHq, 256, false, true);
      const uint32_t tO = tbase + kColO;
      const uint32_t tS = tbase + kColS;
      int g = 0, seg_i = 0;
      bool ok = true;
      // S for global step gs of the current segment (Q resident)
      auto issue_s = [&](int gs) -> bool {
        const int slot = gs % kStages;
        if (!mbar_wait(bar_kv_full(slot), (gs / kStages) & 1, abort_flag, err, kSiteKvFull, gs))
          return false;
        tc_fence_after();
        const uint32_t kb = sStage + slot * kStageBytes;
        for (int a = 0; a < natoms; ++a) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            mma_ss(tS + (gs & 1) * 32, sdesc_sw128(sQ + a * kQAtomBytes + kk * 32, 16, 1024),
                   sdesc_sw128(kb + a * kKAtomBytes + kk * 32, 16, 1024), kIdescS,
                   (a | kk) != 0);
          }
        }
        tc_commit(bar_s_full(gs & 1));
        return true;
      };
      for (int k = cluster; k < nchunks && ok; k += nclusters) {
        ChunkIter it;
        it.init(prefix, B, k, pps, T);
        Seg s;
        while (ok && it.next(s)) {
          const int L = seqlens[s.b];
          const int t0 = s.p0 * kPage, t_end = min(s.p1 * kPage, L);
          const int nsteps = (t_end - t0 + kStep - 1) / kStep;
          ok = mbar_wait(bar_q_full, seg_i & 1, abort_flag, err, kSiteQFull, seg_i);
          if (!ok) break;
          tc_fence_after();
          if (nsteps > 0) ok = issue_s(g);
          if (ok && nsteps > 1) ok = issue_s(g + 1);
          if (ok && nsteps <= 2) tc_commit(bar_q_empty);  // all S of this segment issued
          if (ok && seg_i > 0) {
            ok = mbar_wait(bar_o_free, (seg_i - 1) & 1, abort_flag, err, kSitePvDone, seg_i);
            tc_fence_after();
          }
          for (int i = 0; i < nsteps && ok; ++i) {
            const int gi = g + i;
            ok = mbar_wait(bar_p_full(gi & 1), (gi >> 1) & 1, abort_flag, err, kSitePFull, gi);
            if (!ok) break;
            tc_fence_after();
            const int slot = gi % kStages;
            const uint32_t vb = sStage + slot * kStageBytes;
#pragma unroll
            for (int kk = 0; kk < kStep / 16; ++kk) {
              mma_ts(tO, tS + (gi & 1) * 32 + kk * 8,
                     sdesc_sw128(vb + kk * 16 * 128, kKAtomBytes, 1024), kIdescPV,
                     (i > 0 || kk > 0) ? 1u : 0u);
            }
            tc_commit(bar_kv_empty(slot));
            tc_commit(bar_pv_done);
            if (i + 2 < nsteps) {
              ok = issue_s(gi + 2);
              if (ok && i + 3 == nsteps) tc_commit(bar_q_empty);
            }
          }
          g += nsteps;
          ++seg_i;
        }
      }
      tc_commit(bar_mma_drain);
      volatile int never = 0;
      mbar_wait(bar_mma_drain, 0, &never, nullptr, kSiteDrain, -2);
    }
    __syncwarp();
  } else {
    // ================= softmax, exchange, epilogue (warps 0-3) ============
    const int r = threadIdx.x;  // head == TMEM lane
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t tO = tbase + lane_off + kColO;
    const uint32_t tS = tbase + lane_off + kColS;
    const uint32_t my_x = sX + r * kXRow * 4;
    const uint32_t peer_x = mapa_shared(my_x, peer);
    int g = 0, seg_i = 0;
    bool ok = true;
    for (int k = cluster; k < nchunks && ok; k += nclusters) {
      ChunkIter it;
      it.init(prefix, B, k, pps, T);
      Seg s;
      while (ok && it.next(s)) {
        const int L = seqlens[s.b];
        const int t0 = s.p0 * kPage, t_end = min(s.p1 * kPage, L);
        const int nsteps = (t_end - t0 + kStep - 1) / kStep;
        float m_ref = -INFINITY, l = 0.f;
        for (int i = 0; i < nsteps && ok; ++i) {
          const int gi = g + i, buf = gi & 1, use = gi >> 1;
          ok = mbar_wait(bar_s_full(buf), use & 1, abort_flag, err, kSiteSFull, gi);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
          float sv[kStep];
          tmem_ld32(tS + buf * 32, sv);
          // ---- swap partial S with the peer CTA through DSMEM
          if (use > 0) {
            ok = mbar_wait<true>(bar_xfree(buf), (use - 1) & 1, abort_flag, err, kSiteXfree, gi);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
          }
          const uint32_t dst = peer_x + buf * kXBufBytes;
#pragma unroll
          for (int c = 0; c < kStep; c += 4) st_cluster_v4(dst + c * 4, sv[c], sv[c + 1], sv[c + 2], sv[c + 3]);
          mbar_arrive_cluster(bar_xfull(buf), peer);
          ok = mbar_wait<true>(bar_xfull(buf), use & 1, abort_flag, err, kSiteXchg, gi);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          const float* xin = reinterpret_cast<const float*>(smem + kXOff + buf * kXBufBytes +
                                                            r * kXRow * 4);
#pragma unroll
          for (int c = 0; c < kStep; c += 4) {
            const float4 pv = *reinterpret_cast<const float4*>(xin + c);
            // identical sum order on both CTAs: rank-0 partial + rank-1 partial
            if (rank == 0) {
              sv[c] += pv.x; sv[c + 1] += pv.y; sv[c + 2] += pv.z; sv[c + 3] += pv.w;
            } else {
              sv[c] = pv.x + sv[c]; sv[c + 1] = pv.y + sv[c + 1];
              sv[c + 2] = pv.z + sv[c + 2]; sv[c + 3] = pv.w + sv[c + 3];
            }
          }
          mbar_arrive_cluster(bar_xfree(buf), peer);

          // ---- mask tokens at or past the sequence end, online softmax
          const int tok0 = t0 + i * kStep;
          const int nvalid = L - tok0;
          float mt = -INFINITY;
#pragma unroll
          for (int c = 0; c < kStep; ++c) {
            sv[c] = (c < nvalid) ? sv[c] * scale_log2 : -INFINITY;
            mt = fmaxf(mt, sv[c]);
          }
          const float m_new = fmaxf(m_ref, mt);
          const bool resc = m_new > m_ref + kRescaleThreshold;
          float alpha = 1.f;
          if (resc) {
            alpha = fast_exp2(m_ref - m_new);
            m_ref = m_new;
            l *= alpha;
          }
          const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
          uint32_t p[kStep / 2];
          float rs = 0.f;
#pragma unroll
          for (int c = 0; c < kStep; c += 2) {
            const float p0 = fast_exp2(sv[c] - m_use);
            const float p1 = fast_exp2(sv[c + 1] - m_use);
            rs += p0 + p1;
            p[c / 2] = pack_bf16x2(p0, p1);
          }
          l += rs;
          tmem_st16(tS + buf * 32, p);
          // Tokens past the end contribute exactly zero even if the cache
          // tail holds non-finite bytes: clear those V rows before PV reads.
          if (nvalid < kStep) {
            uint8_t* vst = smem + kStageOff + (gi % kStages) * kStageBytes;
            const int zrows = kStep - nvalid;  // rows [nvalid, 32) of atoms 0..3
            for (int e = threadIdx.x; e < zrows * 4 * 8; e += 128) {
              const int a = e / (zrows * 8), rem = e % (zrows * 8);
              const int rr = nvalid + rem / 8, ch = rem % 8;
              *reinterpret_cast<uint4*>(vst + a * kKAtomBytes + rr * 128 + ch * 16) =
                  make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
            named_barrier_sync(1, 128);
          }
          if (i > 0 && __any_sync(0xffffffffu, resc)) {
            ok = mbar_wait(bar_pv_done, (gi - 1) & 1, abort_flag, err, kSitePvDone, gi);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < 256; c += 32) {
              float ov[32];
              tmem_ld32(tO + c, ov);
              uint32_t ou[32];
#pragma unroll
              for (int t = 0; t < 32; ++t) ou[t] = __float_as_uint(ov[t] * alpha);
              tmem_st32(tO + c, ou);
            }
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(bar_p_full(buf));
        }
        if (!ok) break;
        // ---- segment epilogue
        const int glast = g + nsteps - 1;
        if (nsteps > 0) {
          ok = mbar_wait(bar_pv_done, glast & 1, abort_flag, err, kSitePvDone, glast);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
        }
        const float inv_l = (l > 0.f) ? 1.0f / l : 0.f;
        constexpr float kLn2 = 0.69314718055994530942f;
        const float lse_v = (l > 0.f) ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
        const size_t orow = (size_t)s.b * kHq + r;
#pragma unroll 1
        for (int c = 0; c < 256; c += 32) {
          float ov[32];
          if (nsteps > 0) {
            tmem_ld32(tO + c, ov);
          } else {
#pragma unroll
            for (int t = 0; t < 32; ++t) ov[t] = 0.f;
          }
          if (s.slot < 0) {
            __nv_bfloat16* dst = o + orow * kDv + rank * 256 + c;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              uint4 w;
              w.x = pack_bf16x2(ov[q4 * 8 + 0] * inv_l, ov[q4 * 8 + 1] * inv_l);
              w.y = pack_bf16x2(ov[q4 * 8 + 2] * inv_l, ov[q4 * 8 + 3] * inv_l);
              w.z = pack_bf16x2(ov[q4 * 8 + 4] * inv_l, ov[q4 * 8 + 5] * inv_l);
              w.w = pack_bf16x2(ov[q4 * 8 + 6] * inv_l, ov[q4 * 8 + 7] * inv_l);
              *reinterpret_cast<uint4*>(dst + q4 * 8) = w;
            }
          } else {
            float* dst = part_o + ((size_t)s.slot * kHq + r) * kDv + rank * 256 + c;
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
              *reinterpret_cast<float4*>(dst + q4 * 4) =
                  make_float4(ov[q4 * 4] * inv_l, ov[q4 * 4 + 1] * inv_l,
                              ov[q4 * 4 + 2] * inv_l, ov[q4 * 4 + 3] * inv_l);
          }
        }
        if (rank == 0) {
          if (s.slot < 0) lse[orow] = lse_v;
          else part_lse[(size_t)s.slot * kHq + r] = lse_v;
        }
        tc_fence_before();
        mbar_arrive(bar_o_free);
        g += nsteps;
        ++seg_i;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still touch its smem
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

// ---- combine ------------------------------------------------------------------
// One CTA per (sequence, 16 heads).  Sequences inside one chunk were written
// by the decode kernel; empty sequences get O = 0, LSE = -inf; the rest merge
// their partials: L = log sum_s e^{L_s}, O = sum_s e^{L_s - L} O_s.
__global__ void __launch_bounds__(256) mla_combine_kernel(
    const int* __restrict__ ws_hdr, const int* __restrict__ prefix,
    const float* __restrict__ part_lse, const float* __restrict__ part_o,
    __nv_bfloat16* __restrict__ o, float* __restrict__ lse) {
  const int b = blockIdx.x;
  const int h = blockIdx.y * 16 + (threadIdx.x >> 4);
  const int c0 = (threadIdx.x & 15) * 32;
  const int pps = ws_hdr[1];
  const int pb = prefix[b], pe = prefix[b + 1];
  const size_t orow = (size_t)b * kHq + h;
  if (pe == pb) {
    for (int c = 0; c < 32; c += 8)
      *reinterpret_cast<uint4*>(o + orow * kDv + c0 + c) = make_uint4(0u, 0u, 0u, 0u);
    if (c0 == 0) lse[orow] = -INFINITY;
    return;
  }
  const int k0 = pb / pps, k1 = (pe - 1) / pps;
  if (k0 == k1) return;  // written directly by the decode kernel
  float mx = -INFINITY;
  for (int k = k0; k <= k1; ++k) {
    const int slot = (k == k0 && pb != k0 * pps) ? 2 * k + 1 : 2 * k;
    mx = fmaxf(mx, part_lse[(size_t)slot * kHq + h]);
  }
  float acc[32];
#pragma unroll
  for (int c = 0; c < 32; ++c) acc[c] = 0.f;
  float wsum = 0.f;
  for (int k = k0; k <= k1; ++k) {
    const int slot = (k == k0 && pb != k0 * pps) ? 2 * k + 1 : 2 * k;
    const float ls = part_lse[(size_t)slot * kHq + h];
    const float w = (ls == -INFINITY) ? 0.f : expf(ls - mx);
    wsum += w;
    const float* src = part_o + ((size_t)slot * kHq + h) * kDv + c0;
#pragma unroll
    for (int c = 0; c < 32; c += 4) {
      const float4 v = *reinterpret_cast<const float4*>(src + c);
      acc[c] += w * v.x; acc[c + 1] += w * v.y; acc[c + 2] += w * v.z; acc[c + 3] += w * v.w;
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
  for (int c = 0; c < 32; c += 8) {
    uint4 wv;
    wv.x = pack_bf16x2(acc[c] * inv, acc[c + 1] * inv);
    wv.y = pack_bf16x2(acc[c + 2] * inv, acc[c + 3] * inv);
    wv.z = pack_bf16x2(acc[c + 4] * inv, acc[c + 5] * inv);
    wv.w = pack_bf16x2(acc[c + 6] * inv, acc[c + 7] * inv);
    *reinterpret_cast<uint4*>(o + orow * kDv + c0 + c) = wv;
  }
  if (c0 == 0) lse[orow] = (wsum > 0.f) ? mx + logf(wsum) : -INFINITY;
}

CUresult make_map_2d(CUtensorMap* map, const void* ptr, long long rows, int box_rows) {
  PFN_encodeTiled enc = get_encode_tiled();
  if (!enc) return CUDA_ERROR_NOT_FOUND;
  cuuint64_t dims[2] = {(cuuint64_t)kDk, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kDk * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace

size_t mla_workspace_bytes(int B, int Hq, int max_blocks, int num_sms, int pages_per_split) {
  (void)Hq;
  const int chunks = max_chunks_for(B, max_blocks, num_sms, pages_per_split);
  return ws_layout(B, 2 * chunks).total;
}

cudaError_t launch_mla_decode(const MlaArgs& a, cudaStream_t s) {
  const int clusters = a.num_sms / 2;
  const int max_chunks = max_chunks_for(a.B, a.max_blocks, a.num_sms, a.pages_per_split);
  const WsLayout w = ws_layout(a.B, 2 * max_chunks);
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  int* hdr = reinterpret_cast<int*>(ws + w.header);
  int* prefix = reinterpret_cast<int*>(ws + w.prefix);
  float* plse = reinterpret_cast<float*>(ws + w.plse);
  float* po = reinterpret_cast<float*>(ws + w.po);

  CUtensorMap mq, mkv;
  CUresult r = make_map_2d(&mq, a.q, (long long)a.B * kHq, kHq);
  if (r == CUDA_SUCCESS) r = make_map_2d(&mkv, a.kv, (long long)a.num_blocks * kPage, kStep);
  if (r != CUDA_SUCCESS) {
    attn_set_error("mla_decode: cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return cudaErrorInvalidValue;
  }
  // With a fixed split length the chunk count may exceed the cluster count:
  // clusters then loop over chunks.  The automatic plan makes at most one
  // chunk per cluster.
  mla_plan_kernel<<<1, 1024, 0, s>>>(a.seqlens, a.B, a.max_blocks, clusters, a.pages_per_split,
                                     hdr, prefix, a.err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kSmemBytes);
  if (e != cudaSuccess) return e;
  const float scale_log2 = a.scale * 1.4426950408889634f;
  mla_decode_kernel<<<2 * clusters, kThreads, kSmemBytes, s>>>(
      mq, mkv, a.block_table, a.seqlens, static_cast<__nv_bfloat16*>(a.o), a.lse, hdr, prefix,
      plse, po, a.B, a.max_blocks, a.num_blocks, scale_log2, a.err);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  mla_combine_kernel<<<dim3(a.B, kHq / 16), 256, 0, s>>>(hdr, prefix, plse, po,
                                                         static_cast<__nv_bfloat16*>(a.o), a.lse);
  return cudaGetLastError();
}

// ---- fixed scratch for callers that cannot allocate ---------------------------
// mla_decode_noalloc runs the same plan / decode / combine kernels with the
// workspace placed in this file-scope device array instead of a caller
// buffer.  Its size covers the automatic plan for up to kNoAllocMaxBatch
// sequences on a device of up to kNoAllocMaxSms SMs (2 partial slots per
// 2-SM cluster).  Every GPU that loads the library reserves it until exit.
namespace {
constexpr int kNoAllocMaxBatch = 8192;
constexpr int kNoAllocMaxSms = 160;
constexpr size_t kNoAllocScratchBytes =
    ws_layout(kNoAllocMaxBatch, 2 * (kNoAllocMaxSms / 2)).total;
static_assert(kNoAllocScratchBytes % 256 == 0, "scratch size");

static __device__ __align__(256) uint8_t g_mla_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevs = 64;
void* g_scratch_addr[kMaxDevs] = {};
std::mutex g_scratch_mu;
}  // namespace

int mla_noalloc_max_batch() { return kNoAllocMaxBatch; }
int mla_noalloc_max_sms() { return kNoAllocMaxSms; }

// Device address of the fixed scratch on the current device.  The symbol's
// host-side name is only a stand-in, so the address is looked up with
// cudaGetSymbolAddress once per device (with that device current) and cached.
cudaError_t mla_noalloc_scratch(void** ptr, size_t* bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevs) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_mla_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *ptr = g_scratch_addr[dev];
  *bytes = kNoAllocScratchBytes;
  return cudaSuccess;
}
