// prefill_bf16.cu -- bf16 attention forward on the 5th-generation tensor
// cores (tcgen05 + TMEM), sm_103a.
//
// What it computes is the FlashAttention-2 forward of the "FP32 CUDA-core
// FlashAttention-2 v2" blog (dandandamowang post_1787450400): one Q block is
// resident for the whole KV loop (section 1.2), K/V blocks stream through a
// multi-stage buffer (section 3.2), the softmax is online with a deferred 1/l
// (sections 1.3, 3.3, 3.5), blocks above the causal diagonal are skipped and
// the block crossing it is masked per element (sections 1.4, 3.4).  P is cast
// to bf16 before the PV product, as item 7 of the FlashMLA issue #26 list
// suggests (fp32 -> bf16 conversion of P).
//
// How it maps onto GB300 (nothing here is taken from the pages' Ampere,
// Hopper or RTX kernels):
//   * warp 4  : TMA producer.  Q once, then K_j, V_j into a ring of 32 KB
//               slots (128-byte swizzle), full/empty mbarriers per slot.
//   * warp 5  : MMA issuer (one thread) and TMEM owner.  S_j = Q K_j^T is a
//               tcgen05.mma M=128, N=128, K=D into one of two TMEM S buffers;
//               O += P_j V_j takes P straight from TMEM (the A operand) and V
//               from shared memory, accumulating in TMEM.
//   * warps 0-3: softmax, one thread per query row (TMEM lane = row): load the
//               S row, mask, running max, exp2, row sum, write P (bf16) into
//               the S buffer's columns, rescale O in TMEM only when the max
//               grew by more than 2^8 (lazy rescale; exact because O and l
//               share the stale reference), and finally O/l -> bf16 -> smem ->
//               TMA store, plus LSE.
//   TMEM columns: S0 [0,128), S1 [128,256), O [256, 256+D).
//   Every wait is bounded (about 2 s); a stuck pipeline records
//   ATTN_ERR_DEVICE_TIMEOUT and the CTA unwinds, frees TMEM and exits.
#include <math.h>

#include "common.cuh"

namespace {

using namespace gb300;

constexpr int kBM = 128;              // query rows per CTA
constexpr int kBN = 128;              // keys per KV block
constexpr int kThreads = 192;         // 4 softmax warps + producer + MMA
constexpr int kAtomBytes = 128 * 128; // one 128-row x 64-col bf16 swizzle column
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct Cfg {
  static constexpr int kAtoms = D / 64;
  static constexpr int kTileBytes = kAtoms * kAtomBytes;  // Q, K or V block
  static constexpr int kStages = (D == 128) ? 5 : 8;      // ring slots
  static constexpr int kQOff = 0;
  static constexpr int kRingOff = kTileBytes;
  static constexpr int kBarOff = kRingOff + kStages * kTileBytes;
  // barriers: q_full, kv_full[S], kv_empty[S], s_full[2], p_full[2], pv_done,
  // mma_drain
  static constexpr int kNumBars = 1 + 2 * kStages + 2 + 2 + 1 + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // tmem base, abort flag
  static constexpr int kSmemBytes = kMiscOff + 16 + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS0 = 0;
  static constexpr uint32_t kColO = 256;
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
  auto bar_s_full = [&](int b) { return bar0 + 8u * (1 + 2 * C::kStages + b); };
  auto bar_p_full = [&](int b) { return bar0 + 8u * (3 + 2 * C::kStages + b); };
  const uint32_t bar_pv_done = bar0 + 8u * (5 + 2 * C::kStages);
  const uint32_t bar_mma_drain = bar0 + 8u * (6 + 2 * C::kStages);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work item: heaviest causal Q blocks first across all heads
  const int n_qt = (N + kBM - 1) / kBM;
  const int lin = blockIdx.x;
  const int qt = kCausal ? (n_qt - 1 - lin / BH) : (lin / BH);
  const int bh = lin % BH;
  const int q0 = qt * kBM;
  const int kv_limit = kCausal ? min(q0 + kBM, N) : N;
  const int T = (kv_limit + kBN - 1) / kBN;  // KV blocks visited

  // ---- setup: barriers (thread 0), TMEM (warp 5)
  if (threadIdx.x == 0) {
    mbar_init(bar_q_full, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar_kv_full(s), 1);
      mbar_init(bar_kv_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_s_full(b), 1);
      mbar_init(bar_p_full(b), 128);
    }
    mbar_init(bar_pv_done, 1);
    mbar_init(bar_mma_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    prefetch_tmap(&tmO);
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 4) {
    // ================= TMA producer =================
    if (lane == 0) {
      const uint64_t pol_kv = policy_evict_last();  // K/V are re-read by other Q blocks
      mbar_arrive_expect_tx(bar_q_full, C::kTileBytes);
      for (int a = 0; a < C::kAtoms; ++a)
        tma_load_3d(sQ + a * kAtomBytes, &tmQ, bar_q_full, a * 64, q0, bh);
      int issued_until = 0;  // loads [0, issued_until) were issued
      bool ok = true;
      for (int idx = 0; idx < 2 * T && ok; ++idx) {
        const int slot = idx % C::kStages;
        const int use = idx / C::kStages;
        if (use > 0) {
          ok = mbar_wait(bar_kv_empty(slot), (use - 1) & 1, abort_flag, err, kSiteKvEmpty,
                         idx);
          if (!ok) break;
        }
        if (debug_skip_load > 0 && idx == debug_skip_load) continue;  // test hook
        const int j = idx >> 1;
        const CUtensorMap* m = (idx & 1) ? &tmV : &tmK;
        const uint32_t dst = sRing + slot * C::kTileBytes;
        mbar_arrive_expect_tx(bar_kv_full(slot), C::kTileBytes);
        for (int a = 0; a < C::kAtoms; ++a)
          tma_load_3d_hint(dst + a * kAtomBytes, m, bar_kv_full(slot), a * 64, j * kBN, bh,
                           pol_kv);
        issued_until = idx + 1;
      }
      if (!ok) {
        // Let every copy this thread started land before the CTA unwinds.
        const int first = issued_until > C::kStages ? issued_until - C::kStages : 0;
        for (int idx = first; idx < issued_until; ++idx) {
          if (debug_skip_load > 0 && idx == debug_skip_load) continue;
          const int slot = idx % C::kStages;
          volatile int never = 0;
          mbar_wait(bar_kv_full(slot), (idx / C::kStages) & 1, &never, nullptr, kSiteDrain,
                    idx);
        }
        volatile int never = 0;
        mbar_wait(bar_q_full, 0, &never, nullptr, kSiteDrain, -1);
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ================= MMA issuer =================
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_bf16(kBM, kBN, false, false);
      constexpr uint32_t kIdescPV = idesc_bf16(kBM, D, false, true);
      const uint32_t tS = tbase + C::kColS0;
      const uint32_t tO = tbase + C::kColO;
      bool ok = mbar_wait(bar_q_full, 0, abort_flag, err, kSiteQFull, 0);
      tc_fence_after();

      auto issue_s = [&](int j) -> bool {
        const int idx = 2 * j;
        const int slot = idx % C::kStages;
        if (!mbar_wait(bar_kv_full(slot), (idx / C::kStages) & 1, abort_flag, err,
                       kSiteKvFull, idx))
          return false;
        tc_fence_after();
        const uint32_t kb = sRing + slot * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kAtomBytes + (kk & 3) * 32;
          mma_ss(tS + (j & 1) * 128, sdesc_sw128(sQ + off, 16, 1024),
                 sdesc_sw128(kb + off, 16, 1024), kIdescS, kk > 0);
        }
        tc_commit(bar_kv_empty(slot));
        tc_commit(bar_s_full(j & 1));
        return true;
      };

      if (ok) ok = issue_s(0);
      if (ok && T > 1) ok = issue_s(1);
      for (int j = 0; j < T && ok; ++j) {
        ok = mbar_wait(bar_p_full(j & 1), (j >> 1) & 1, abort_flag, err, kSitePFull, j);
        if (!ok) break;
        tc_fence_after();
        const int idx = 2 * j + 1;
        const int slot = idx % C::kStages;
        ok = mbar_wait(bar_kv_full(slot), (idx / C::kStages) & 1, abort_flag, err,
                       kSiteKvFull, idx);
        if (!ok) break;
        tc_fence_after();
        const uint32_t vb = sRing + slot * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          // A = P (bf16, 2 per TMEM column): keys [16kk, 16kk+16) = 8 columns.
          // B = V block, MN-major: 16 keys = 2 groups of 8 rows of 128 B.
          mma_ts(tO, tS + (j & 1) * 128 + kk * 8,
                 sdesc_sw128(vb + kk * 16 * 128, kAtomBytes, 1024), kIdescPV,
                 (j > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(bar_kv_empty(slot));
        tc_commit(bar_pv_done);
        if (j + 2 < T) ok = issue_s(j + 2);
      }
      // Every MMA this thread issued must be complete before TMEM is freed.
      tc_commit(bar_mma_drain);
      volatile int never = 0;
      mbar_wait(bar_mma_drain, 0, &never, nullptr, kSiteDrain, -2);
    }
    __syncwarp();
  } else {
    // ================= softmax + correction + epilogue (warps 0-3) =========
    const int r = threadIdx.x;  // row within the Q block == TMEM lane
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t tS = tbase + lane_off + C::kColS0;
    const uint32_t tO = tbase + lane_off + C::kColO;
    const int row = q0 + r;
    // keys [0, lim) are visible to this row
    const int lim = kCausal ? min(N, row + 1) : N;
    float m_ref = -INFINITY;  // running max (log2 units), lazily updated
    float l = 0.f;
    bool ok = true;

    for (int j = 0; j < T; ++j) {
      ok = mbar_wait(bar_s_full(j & 1), (j >> 1) & 1, abort_flag, err, kSiteSFull, j);
      ok = __all_sync(0xffffffffu, ok);  // tcgen05.ld/st below are warp-collective
      if (!ok) break;
      tc_fence_after();
      float s[kBN];
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c) tmem_ld32(tS + (j & 1) * 128 + c * 32, s + c * 32);

      const int kv0 = j * kBN;
      const int nvalid = lim - kv0;  // keys k < nvalid of this block are visible
      float mt = -INFINITY;
      if (nvalid >= kBN) {
#pragma unroll
        for (int c = 0; c < kBN; ++c) {
          s[c] *= scale_log2;
          mt = fmaxf(mt, s[c]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < kBN; ++c) {
          s[c] = (c < nvalid) ? s[c] * scale_log2 : -INFINITY;
          mt = fmaxf(mt, s[c]);
        }
      }
      const float m_new = fmaxf(m_ref, mt);
      const bool resc = m_new > m_ref + kRescaleThreshold;  // false while both -inf
      float alpha = 1.f;
      if (resc) {
        alpha = fast_exp2(m_ref - m_new);  // 0 when m_ref == -inf
        m_ref = m_new;
        l *= alpha;
      }
      const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
      uint32_t p[kBN / 2];
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < kBN; c += 2) {
        const float p0 = fast_exp2(s[c] - m_use);
        const float p1 = fast_exp2(s[c + 1] - m_use);
        rs += p0 + p1;
        p[c / 2] = pack_bf16x2(p0, p1);
      }
      l += rs;
#pragma unroll
      for (int c = 0; c < kBN / 64; ++c) tmem_st32(tS + (j & 1) * 128 + c * 32, p + c * 32);

      // Lazy correction of O: needed only if some row of this warp moved its
      // reference, and only once PV_{j-1} has landed in TMEM.
      if (j > 0 && __any_sync(0xffffffffu, resc)) {
        ok = mbar_wait(bar_pv_done, (j - 1) & 1, abort_flag, err, kSitePvDone, j);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          float ov[32];
          tmem_ld32(tO + c * 32, ov);
          uint32_t ou[32];
#pragma unroll
          for (int t = 0; t < 32; ++t) ou[t] = __float_as_uint(ov[t] * alpha);
          tmem_st32(tO + c * 32, ou);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar_p_full(j & 1));
    }

    if (ok) ok = mbar_wait(bar_pv_done, (T - 1) & 1, abort_flag, err, kSitePvDone, T);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      tc_fence_after();
      // ---- epilogue: O / l -> bf16 into the (now free) Q buffer, TMA store
      const float inv_l = 1.0f / l;
      uint8_t* stage = smem + C::kQOff;
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
    // All four softmax warps reach this barrier on every path (their waits
    // are bounded); the store is skipped if any role aborted.
    named_barrier_sync(1, 128);
    if (threadIdx.x == 0 && *abort_flag == 0) {
      for (int a = 0; a < C::kAtoms; ++a) tma_store_3d(&tmO, sQ + a * kAtomBytes, a * 64, q0, bh);
      bulk_commit();
      bulk_wait_all();
    }
  }

  // ---- teardown: every role has finished (or unwound); free TMEM
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
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

template <int D, bool kCausal>
cudaError_t launch_t(const PrefillBf16Args& a, const CUtensorMap& mq, const CUtensorMap& mk,
                     const CUtensorMap& mv, const CUtensorMap& mo, cudaStream_t s) {
  using C = Cfg<D>;
  auto kern = prefill_bf16_kernel<D, kCausal>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int BH = a.B * a.H;
  const long long blocks = (long long)((a.N + kBM - 1) / kBM) * BH;
  const float scale_log2 = a.scale * 1.4426950408889634f;
  kern<<<(unsigned)blocks, kThreads, C::kSmemBytes, s>>>(mq, mk, mv, mo, a.lse, BH, a.N,
                                                          scale_log2, a.err, a.debug_skip_load);
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
  const int BH = a.B * a.H;
  const long long blocks = (long long)((a.N + kBM - 1) / kBM) * BH;
  if (blocks > 0x7fffffffLL) {
    attn_set_error("attn_fwd: too many query blocks (%lld)", blocks);
    return cudaErrorInvalidValue;
  }
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
