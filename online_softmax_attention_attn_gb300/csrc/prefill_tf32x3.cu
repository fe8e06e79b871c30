// prefill_tf32x3.cu -- fp32 attention forward on the 5th-generation tensor
// cores with the three-product TF32 split ("3xTF32"), sm_103a.
//
// What it computes is the fp32 FlashAttention-2 forward of the "FP32
// CUDA-core FlashAttention-2 v2" blog (dandandamowang post_1787450400): a Q
// block of 128 rows stays on chip for the whole KV loop (section 1.2), the
// softmax is online with a deferred 1/l (sections 1.3, 3.3, 3.5), blocks above
// the causal diagonal are skipped and the blocks crossing it are masked per
// element (sections 1.4, 3.4).  The blog names tensor cores as the step it has
// not taken yet (section 5); its workload (section 4.1: B4 H8 N8192 D64,
// fp32) is the one this kernel is measured on.
//
// fp32 accuracy from TF32 MMAs.  A TF32 operand keeps 10 explicit mantissa
// bits, too few for a 1e-4 bound on O.  Each fp32 operand x is written as
// x = hi + lo with hi = x rounded to TF32 and lo = (x - hi) rounded to TF32;
// then x*y ~ lo_x*hi_y + hi_x*lo_y + hi_x*hi_y, the dropped lo_x*lo_y and the
// rounding of lo being below 2^-21 |x*y|.  Q K^T is three tcgen05.mma
// kind::tf32 into one fp32 accumulator.  In P V the two cross terms carry
// only 2^-11 of the product, so they run as kind::f16 MMAs on bf16 operands
// (bf16(P_lo) bf16(V) + bf16(P) bf16(V_lo), 16 keys per MMA instead of 8)
// into the same fp32 accumulator: their bf16 rounding costs below 2^-19 of
// each product, against a bound of 1e-4 on O, and P V needs 16 MMAs per
// block instead of 24.
//
// Layout and roles (one Q tile of 128 rows per CTA, 224 threads):
//   * pre-pass (tf32x3_split_kernel): K -> K_hi, K_lo ([BH, N, 64] fp32) and
//     V -> V^T_hi (fp32), bf16(V)^T and bf16(V_lo)^T ([BH, 64, Np], Np = N
//     rounded up to 64, tail keys zero) in a caller workspace, once per call,
//     so that every MMA operand is K-major (the keys are the contraction
//     dimension of P V).
//   * warp 4 : TMA producer.  K_hi, K_lo, V^T_hi (16 KB each) and the two
//     bf16 V^T tiles (8 KB each) of one 64-key block form one 64 KB stage
//     (128-byte swizzle); 3 stages.
//   * warp 6 : S issuer (one thread).
//       S_j = Q K_j^T : A = Q_hi / Q_lo from TMEM, B = K_hi / K_lo (smem),
//                       M=128 N=64, 8 k-steps of 8 x 3 products,
//     into buffer j&1 once PV_{j-2} (the last reader of that buffer) is done.
//   * warp 5 : PV issuer (one thread) and TMEM owner.
//       O += P_j V_j  : hi x hi: A = P_hi (tf32, TMEM), B = V^T_hi, 8 k-steps
//                       of 8; cross terms: A = bf16(P_lo) / bf16(P) (TMEM),
//                       B = bf16(V)^T / bf16(V_lo)^T, 4 k-steps of 16 x 2.
//     Two S buffers keep the tensor core busy while the softmax of the other
//     block runs; two issuing threads in different warps keep the pipe fed
//     (one thread alone is paced by its own issue cost, not by the pipe).
//   * warps 0-3 : softmax, one thread per query row (TMEM lane = row).  They
//     split the row's Q into TMEM, then per block: S -> scale, mask, running
//     max (lazy: O and l are rescaled only when the max grew by more than
//     2^8, exact because both share the stale reference), P = 2^(t - m),
//     row sum, P_hi over the S columns, bf16(P) and bf16(P_lo) beside them.
//     Epilogue:
//     O / l (fp32) and LSE straight to global memory.
//   TMEM columns: Q_hi [0,64), Q_lo [64,128), O [128,192),
//   buffer b: S / P_hi [256+128b, +64), bf16(P) [320+128b, +32),
//   bf16(P_lo) [352+128b, +32) (two bf16 per column).
//   Every wait is bounded (about 2 s); a stuck pipeline records
//   ATTN_ERR_DEVICE_TIMEOUT and the CTA unwinds, frees TMEM and exits.
#include <math.h>

#include "common.cuh"

namespace {

using namespace gb300;

constexpr int kD = 64;
constexpr int kBM = 128;               // query rows per CTA
constexpr int kBN = 64;                // keys per KV block
constexpr int kThreads = 224;          // 4 softmax warps, producer, PV issuer, S issuer
constexpr int kAtomBytes = 64 * 128;   // 64 rows x 128 B (one 128-byte swizzle column)
constexpr int kPartBytes = 2 * kAtomBytes;  // one 64 x 64 fp32 operand block
constexpr int kVbOff = 3 * kPartBytes;      // bf16(V)^T: one atom (64 rows x 64 bf16)
constexpr int kVlbOff = kVbOff + kAtomBytes;  // bf16(V_lo)^T
constexpr int kStageBytes = kVlbOff + kAtomBytes;  // K_hi, K_lo, V^T_hi, two bf16 V^T
constexpr int kStages = 3;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kHeadGroup = 4;              // heads whose tiles are scheduled together

constexpr int kRingOff = 0;
constexpr int kBarOff = kRingOff + kStages * kStageBytes;
// barriers: q_full, kv_full[S], kv_empty[S], s_full[2], p_full[2],
// pv_done[2], pv_drain, s_drain.  The two-buffer barriers complete once every
// other block, so no waiter is ever two of their phases behind or ahead.
constexpr int kNumBars = 1 + 2 * kStages + 2 + 2 + 2 + 2;
constexpr int kMiscOff = kBarOff + kNumBars * 8;  // tmem base, abort flag
constexpr int kSmemBytes = kMiscOff + 16 + 1024;  // + alignment slack
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColQhi = 0;
constexpr uint32_t kColQlo = 64;
constexpr uint32_t kColO = 128;
constexpr uint32_t kColS = 256;    // + 128 * buffer; bf16(P) at + 64, bf16(P_lo) at + 96

// Round to the TF32 grid (10 explicit mantissa bits), to nearest with ties
// away from zero: add half a TF32 unit to the magnitude bits and clear the 13
// low bits.  Finite inputs of magnitude below 2^127 only.
__device__ __forceinline__ float tf32_round(float x) {
  return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xFFFFE000u);
}

// ------------------------------------------------------------ pre-pass

// One block per 64 keys, looping over heads: K rows are split in place of
// layout, V rows split (V_hi in fp32, V and V - V_hi in bf16) and transposed
// through shared memory.  Keys in
// [N, Np) of V^T are written as zeros (their P is 0, and 0 * garbage could
// be NaN); K rows past N are never read (the tensor map ends at N).
__device__ __forceinline__ void split4(float4 x, float4& h, float4& l) {
  h.x = tf32_round(x.x); l.x = tf32_round(x.x - h.x);
  h.y = tf32_round(x.y); l.y = tf32_round(x.y - h.y);
  h.z = tf32_round(x.z); l.z = tf32_round(x.z - h.z);
  h.w = tf32_round(x.w); l.w = tf32_round(x.w - h.w);
}

__global__ void __launch_bounds__(256)
    tf32x3_split_kernel(const float* __restrict__ k, const float* __restrict__ v,
                        float* __restrict__ k_hi, float* __restrict__ k_lo,
                        float* __restrict__ vt_hi, __nv_bfloat16* __restrict__ vt_b,
                        __nv_bfloat16* __restrict__ vt_lo_b, int N, int Np, int BH) {
  __shared__ float tile[64][kD + 1];
  // the attention kernel may be scheduled now; it waits for this grid's
  // completion before its first read of the split operands
  grid_launch_dependents();
  const int key0 = blockIdx.x * 64;
  for (int bh = blockIdx.y; bh < BH; bh += gridDim.y) {
    const size_t row_base = (size_t)bh * N;
    // K and V: 64 rows x 16 float4, 4 per thread
    for (int i = threadIdx.x; i < 64 * 16; i += 256) {
      const int r = i >> 4, c4 = i & 15;
      const int key = key0 + r;
      float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
      if (key < N) {
        const size_t off = (row_base + key) * kD + 4 * c4;
        float4 h, l;
        split4(*reinterpret_cast<const float4*>(k + off), h, l);
        *reinterpret_cast<float4*>(k_hi + off) = h;
        *reinterpret_cast<float4*>(k_lo + off) = l;
        y = *reinterpret_cast<const float4*>(v + off);
      }
      tile[r][4 * c4 + 0] = y.x;
      tile[r][4 * c4 + 1] = y.y;
      tile[r][4 * c4 + 2] = y.z;
      tile[r][4 * c4 + 3] = y.w;
    }
    __syncthreads();
    // V^T: 64 d-rows x 16 float4 of keys
    const size_t vt_base = (size_t)bh * kD * Np;
    for (int i = threadIdx.x; i < 64 * 16; i += 256) {
      const int d = i >> 4, k4 = i & 15;
      const float4 x = make_float4(tile[4 * k4][d], tile[4 * k4 + 1][d], tile[4 * k4 + 2][d],
                                   tile[4 * k4 + 3][d]);
      float4 h, l;
      split4(x, h, l);
      const size_t off = vt_base + (size_t)d * Np + key0 + 4 * k4;
      *reinterpret_cast<float4*>(vt_hi + off) = h;
      // the cross terms' bf16 operands: V itself and V - V_hi
      *reinterpret_cast<uint2*>(vt_b + off) =
          make_uint2(pack_bf16x2(x.x, x.y), pack_bf16x2(x.z, x.w));
      *reinterpret_cast<uint2*>(vt_lo_b + off) = make_uint2(
          pack_bf16x2(x.x - h.x, x.y - h.y), pack_bf16x2(x.z - h.z, x.w - h.w));
    }
    __syncthreads();  // the tile is refilled for the next head
  }
}

// ------------------------------------------------------------ attention

template <bool kCausal>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tf32x3_kernel(const __grid_constant__ CUtensorMap tmKhi,
                          const __grid_constant__ CUtensorMap tmKlo,
                          const __grid_constant__ CUtensorMap tmVhi,
                          const __grid_constant__ CUtensorMap tmVb,
                          const __grid_constant__ CUtensorMap tmVlb,
                          const float* __restrict__ q, float* __restrict__ o,
                          float* __restrict__ lse, int BH, int N, float scale_log2, int* err,
                          int debug_skip_block) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment: swizzle atoms must start on a 1024-byte boundary.
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);

  const uint32_t sRing = base + kRingOff;
  const uint32_t bar0 = base + kBarOff;
  const uint32_t bar_q_full = bar0;
  auto bar_kv_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto bar_kv_empty = [&](int s) { return bar0 + 8u * (1 + kStages + s); };
  auto bar_s_full = [&](int b) { return bar0 + 8u * (1 + 2 * kStages + b); };
  auto bar_p_full = [&](int b) { return bar0 + 8u * (3 + 2 * kStages + b); };
  auto bar_pv_done = [&](int b) { return bar0 + 8u * (5 + 2 * kStages + b); };
  const uint32_t bar_pv_drain = bar0 + 8u * (7 + 2 * kStages);
  const uint32_t bar_s_drain = bar0 + 8u * (8 + 2 * kStages);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kMiscOff + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Blocks run in launch order, in groups of kHeadGroup heads: the CTAs in
  // flight share one group's split K/V in L2 (8 MB per head at N = 8192, so
  // 32 MB per group; groups of 8 heads let part of it be evicted before its
  // last reader and read K/V from DRAM again).
  // Within a group the heaviest causal tiles come first, across its heads.
  const int n_qt = (N + kBM - 1) / kBM;
  const int group = (int)(blockIdx.x / (unsigned)(kHeadGroup * n_qt));
  const int g_heads = min(kHeadGroup, BH - group * kHeadGroup);
  const int rem = (int)blockIdx.x - group * kHeadGroup * n_qt;
  const int bh = group * kHeadGroup + rem % g_heads;
  const int qt = kCausal ? n_qt - 1 - rem / g_heads : rem / g_heads;
  const int q0 = qt * kBM;
  const int kv_limit = kCausal ? min(q0 + kBM, N) : N;
  const int T = (kv_limit + kBN - 1) / kBN;  // >= 1

  // ---- setup: barriers (thread 0), TMEM (warp 5)
  if (threadIdx.x == 0) {
    mbar_init(bar_q_full, 128);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_kv_full(s), 1);
      mbar_init(bar_kv_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_s_full(b), 1);
      mbar_init(bar_p_full(b), 128);
      mbar_init(bar_pv_done(b), 1);
    }
    mbar_init(bar_pv_drain, 1);
    mbar_init(bar_s_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmKhi);
    prefetch_tmap(&tmKlo);
    prefetch_tmap(&tmVhi);
    prefetch_tmap(&tmVb);
    prefetch_tmap(&tmVlb);
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 4) {
    // ================= TMA producer =================
    if (lane == 0) {
      // the split operands are written by the pre-pass grid
      grid_dependency_wait();
      const uint64_t pol = policy_evict_last();  // re-read by the head's other Q tiles
      bool ok = true;
      int j = 0;
      for (; j < T; ++j) {
        const int s = j % kStages;
        const int use = j / kStages;
        if (use > 0) {
          ok = mbar_wait(bar_kv_empty(s), (use - 1) & 1, abort_flag, err, kSiteKvEmpty, j);
          if (!ok) break;
        }
        if (j == debug_skip_block) continue;  // test hook: this block never arrives
        const uint32_t dst = sRing + s * kStageBytes;
        const uint32_t bar = bar_kv_full(s);
        mbar_arrive_expect_tx(bar, kStageBytes);
#pragma unroll
        for (int a = 0; a < 2; ++a) {
          tma_load_3d_hint(dst + a * kAtomBytes, &tmKhi, bar, 32 * a, j * kBN, bh, pol);
          tma_load_3d_hint(dst + kPartBytes + a * kAtomBytes, &tmKlo, bar, 32 * a, j * kBN, bh,
                           pol);
          tma_load_3d_hint(dst + 2 * kPartBytes + a * kAtomBytes, &tmVhi, bar, j * kBN + 32 * a,
                           0, bh, pol);
        }
        tma_load_3d_hint(dst + kVbOff, &tmVb, bar, j * kBN, 0, bh, pol);
        tma_load_3d_hint(dst + kVlbOff, &tmVlb, bar, j * kBN, 0, bh, pol);
      }
      if (!ok) {
        // let every copy this thread started land before the CTA unwinds
        const int first = j > kStages ? j - kStages : 0;
        for (int x = first; x < j; ++x) {
          if (x == debug_skip_block) continue;
          volatile int never = 0;
          mbar_wait(bar_kv_full(x % kStages), (x / kStages) & 1, &never, nullptr, kSiteDrain,
                    x);
        }
      }
    }
    __syncwarp();
  } else if (warp == 5 || warp == 6) {
    // ================= MMA issuers: PV (warp 5), S (warp 6) =================
    if (lane == 0) {
      constexpr uint32_t kIdesc = idesc_tf32(kBM, 64);
      constexpr uint32_t kIdescB = idesc_bf16(kBM, 64, false, false);
      // K-major operands, 128-byte rows of 32 floats in 8-row groups 1024 B
      // apart; a k-step of 8 floats is 32 B inside the atom, the second half
      // of the 64-wide contraction is the next atom.
      const uint64_t d0 = sdesc_sw128(sRing, 16, 1024);
      bool ok = true;
      if (warp == 6) {
        ok = mbar_wait(bar_q_full, 0, abort_flag, err, kSiteQFull, 0);
        for (int j = 0; j < T && ok; ++j) {
          const int s = j % kStages;
          // buffer j&1 was last read by PV_{j-2}
          if (j >= 2)
            ok = mbar_wait(bar_pv_done(j & 1), ((j - 2) >> 1) & 1, abort_flag, err,
                           kSitePvDone, j);
          if (ok) ok = mbar_wait(bar_kv_full(s), (j / kStages) & 1, abort_flag, err,
                                 kSiteKvFull, j);
          if (!ok) break;
          tc_fence_after();
          const uint32_t dS = tbase + kColS + 128u * (j & 1);
          const uint64_t khi = d0 + (uint64_t)((s * kStageBytes) >> 4);
          const uint64_t klo = khi + (uint64_t)(kPartBytes >> 4);
#pragma unroll
          for (int kk = 0; kk < kD / 8; ++kk) {
            const uint64_t off = (uint64_t)(((kk >> 2) * kAtomBytes + (kk & 3) * 32) >> 4);
            mma_ts_tf32(dS, tbase + kColQlo + 8 * kk, khi + off, kIdesc, kk > 0);
            mma_ts_tf32(dS, tbase + kColQhi + 8 * kk, klo + off, kIdesc, 1u);
            mma_ts_tf32(dS, tbase + kColQhi + 8 * kk, khi + off, kIdesc, 1u);
          }
          tc_commit(bar_s_full(j & 1));
        }
        // every MMA this thread issued must be complete before TMEM is freed
        tc_commit(bar_s_drain);
        volatile int never = 0;
        mbar_wait(bar_s_drain, 0, &never, nullptr, kSiteDrain, -3);
      } else {
        for (int j = 0; j < T && ok; ++j) {
          const int b = j & 1;
          ok = mbar_wait(bar_p_full(b), (j >> 1) & 1, abort_flag, err, kSitePFull, j);
          if (!ok) break;
          tc_fence_after();
          const int s = j % kStages;
          const uint64_t vhi = d0 + (uint64_t)((s * kStageBytes + 2 * kPartBytes) >> 4);
          const uint64_t vb = d0 + (uint64_t)((s * kStageBytes + kVbOff) >> 4);
          const uint64_t vlb = d0 + (uint64_t)((s * kStageBytes + kVlbOff) >> 4);
          const uint32_t aPhi = tbase + kColS + 128u * b;
          const uint32_t aPb = aPhi + 64;
          const uint32_t aPlb = aPhi + 96;
          const uint32_t dO = tbase + kColO;
          // cross terms first (bf16, 16 keys = 8 columns = 32 B per k-step)
#pragma unroll
          for (int kb = 0; kb < kBN / 16; ++kb) {
            const uint64_t off = (uint64_t)((kb * 32) >> 4);
            mma_ts(dO, aPlb + 8 * kb, vb + off, kIdescB, (j > 0 || kb > 0) ? 1u : 0u);
            mma_ts(dO, aPb + 8 * kb, vlb + off, kIdescB, 1u);
          }
#pragma unroll
          for (int kk = 0; kk < kBN / 8; ++kk) {
            const uint64_t off = (uint64_t)(((kk >> 2) * kAtomBytes + (kk & 3) * 32) >> 4);
            mma_ts_tf32(dO, aPhi + 8 * kk, vhi + off, kIdesc, 1u);
          }
          tc_commit(bar_pv_done(b));
          // S_j completed before P_j existed, so PV_j is the stage's last reader
          tc_commit(bar_kv_empty(s));
        }
        tc_commit(bar_pv_drain);
        volatile int never = 0;
        mbar_wait(bar_pv_drain, 0, &never, nullptr, kSiteDrain, -2);
      }
    }
    __syncwarp();
  } else {
    // ================= softmax warps 0-3 =================
    const int r = threadIdx.x;  // row within the tile == TMEM lane
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const int row = q0 + r;
    const int lim = kCausal ? min(N, row + 1) : N;  // keys [0, lim) are visible
    const size_t grow = (size_t)bh * N + row;

    // Q row -> Q_hi, Q_lo in TMEM (rows past N are zero)
    {
      float qv[kD];
      if (row < N) {
#pragma unroll
        for (int c = 0; c < kD; c += 4) {
          const float4 x = *reinterpret_cast<const float4*>(q + grow * kD + c);
          qv[c] = x.x; qv[c + 1] = x.y; qv[c + 2] = x.z; qv[c + 3] = x.w;
        }
      } else {
#pragma unroll
        for (int c = 0; c < kD; ++c) qv[c] = 0.f;
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t hi[32], lo[32];
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          const float x = qv[32 * h + u];
          const float xh = tf32_round(x);
          hi[u] = __float_as_uint(xh);
          lo[u] = __float_as_uint(tf32_round(x - xh));
        }
        tmem_st32(tbase + lane_off + kColQhi + 32 * h, hi);
        tmem_st32(tbase + lane_off + kColQlo + 32 * h, lo);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar_q_full);
    }

    float m_ref = -INFINITY;  // running max (log2 units), lazily updated
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < T; ++j) {
      const int b = j & 1;
      ok = mbar_wait(bar_s_full(b), (j >> 1) & 1, abort_flag, err, kSiteSFull, j);
      ok = __all_sync(0xffffffffu, ok);  // tcgen05.ld/st below are warp-collective
      if (!ok) break;
      tc_fence_after();
      const uint32_t tS = tbase + lane_off + kColS + 128u * b;
      float sv[kBN];
      tmem_ld64(tS, sv);
      const int nvalid = lim - j * kBN;  // keys c < nvalid of this block are visible
      float mt = -INFINITY;
#pragma unroll
      for (int c = 0; c < kBN; ++c) {
        sv[c] = (c < nvalid) ? sv[c] * scale_log2 : -INFINITY;
        mt = fmaxf(mt, sv[c]);
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
      float r0 = 0.f, r1 = 0.f, r2 = 0.f, r3 = 0.f;
#pragma unroll
      for (int c = 0; c < kBN; c += 4) {
        sv[c] = fast_exp2(sv[c] - m_use);
        sv[c + 1] = fast_exp2(sv[c + 1] - m_use);
        sv[c + 2] = fast_exp2(sv[c + 2] - m_use);
        sv[c + 3] = fast_exp2(sv[c + 3] - m_use);
        r0 += sv[c]; r1 += sv[c + 1]; r2 += sv[c + 2]; r3 += sv[c + 3];
      }
      l += (r0 + r1) + (r2 + r3);
      // P_hi (tf32) over the S columns; bf16(P) and bf16(P - P_hi) beside them
      {
        uint32_t pb[32], plb[32];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t hi[32];
#pragma unroll
          for (int u = 0; u < 32; u += 2) {
            const float x0 = sv[32 * h + u], x1 = sv[32 * h + u + 1];
            const float h0 = tf32_round(x0), h1 = tf32_round(x1);
            hi[u] = __float_as_uint(h0);
            hi[u + 1] = __float_as_uint(h1);
            pb[16 * h + u / 2] = pack_bf16x2(x0, x1);
            plb[16 * h + u / 2] = pack_bf16x2(x0 - h0, x1 - h1);
          }
          tmem_st32(tS + 32 * h, hi);
        }
        tmem_st32(tS + 64, pb);
        tmem_st32(tS + 96, plb);
      }
      // Lazy correction of O before PV_j: only if some row of this warp moved
      // its reference, and only once PV_{j-1} has landed.
      if (j > 0 && __any_sync(0xffffffffu, resc)) {
        ok = mbar_wait(bar_pv_done((j - 1) & 1), ((j - 1) >> 1) & 1, abort_flag, err,
                       kSitePvDone, j);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < kD; c += 32) {
          float ov[32];
          tmem_ld32(tbase + lane_off + kColO + c, ov);
          uint32_t ou[32];
#pragma unroll
          for (int u = 0; u < 32; ++u) ou[u] = __float_as_uint(ov[u] * alpha);
          tmem_st32(tbase + lane_off + kColO + c, ou);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar_p_full(b));
    }

    // ---- epilogue: O / l and LSE straight to global memory
    if (ok)
      ok = mbar_wait(bar_pv_done((T - 1) & 1), ((T - 1) >> 1) & 1, abort_flag, err,
                     kSitePvDone, T);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      tc_fence_after();
      float ov[kD];
      tmem_ld64(tbase + lane_off + kColO, ov);
      if (row < N) {
        const float inv_l = 1.0f / l;
#pragma unroll
        for (int c = 0; c < kD; c += 4) {
          float4 w = make_float4(ov[c] * inv_l, ov[c + 1] * inv_l, ov[c + 2] * inv_l,
                                 ov[c + 3] * inv_l);
          *reinterpret_cast<float4*>(o + grow * kD + c) = w;
        }
        constexpr float kLn2 = 0.69314718055994530942f;
        lse[grow] = (m_ref + log2f(l)) * kLn2;
      }
    }
  }

  // ---- teardown: every role has finished (or unwound); free TMEM
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

// Tensor maps over the split operands: K parts [BH, N, 64] with boxes of
// 32 floats x 64 keys, V^T parts [BH, 64, Np] with boxes of 128 bytes of keys
// (32 fp32 or 64 bf16) x 64 rows.
CUresult make_map(CUtensorMap* map, const void* ptr, cuuint64_t inner, cuuint64_t rows, int BH,
                  int esize) {
  PFN_encodeTiled enc = get_encode_tiled();
  if (!enc) return CUDA_ERROR_NOT_FOUND;
  cuuint64_t dims[3] = {inner, rows, (cuuint64_t)BH};
  cuuint64_t strides[2] = {inner * esize, inner * rows * esize};
  cuuint32_t box[3] = {(cuuint32_t)(128 / esize), 64, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, esize == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
             3, const_cast<void*>(ptr), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

struct WsParts {
  size_t k_bytes, vt_bytes, total;  // vt_bytes: the fp32 V^T_hi part
  int Np;
};

WsParts ws_parts(int B, int H, int N) {
  WsParts w;
  const size_t BH = (size_t)B * H;
  w.Np = (N + 63) / 64 * 64;
  w.k_bytes = BH * (size_t)N * kD * 4;
  w.k_bytes = (w.k_bytes + 255) / 256 * 256;
  w.vt_bytes = BH * (size_t)kD * w.Np * 4;
  w.total = 2 * w.k_bytes + 2 * w.vt_bytes;  // V^T_hi, then two bf16 parts of half its size
  return w;
}

template <bool kCausal>
cudaError_t launch_t(const PrefillTf32x3Args& a, const CUtensorMap* maps, float scale_log2,
                     cudaStream_t s) {
  auto kern = prefill_tf32x3_kernel<kCausal>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBytes);
  if (e != cudaSuccess) return e;
  const int BH = a.B * a.H;
  const long long tiles = (long long)BH * ((a.N + kBM - 1) / kBM);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)tiles);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], maps[3], maps[4], a.q, a.o,
                            a.lse, BH, a.N, scale_log2, a.err, a.debug_skip_block);
}

}  // namespace

size_t prefill_tf32x3_workspace_bytes(int B, int H, int N) { return ws_parts(B, H, N).total; }

bool prefill_tf32x3_info(int* Br, int* Bc, int* threads, int* smem) {
  if (Br) *Br = kBM;
  if (Bc) *Bc = kBN;
  if (threads) *threads = kThreads;
  if (smem) *smem = kSmemBytes;
  return true;
}

cudaError_t launch_prefill_tf32x3(const PrefillTf32x3Args& a, cudaStream_t s) {
  const int BH = a.B * a.H;
  const long long tiles = (long long)BH * ((a.N + kBM - 1) / kBM);
  if (tiles > 0x7fffffffLL) {
    attn_set_error("attn_fwd_tf32x3: too many query tiles (%lld)", tiles);
    return cudaErrorInvalidValue;
  }
  const WsParts w = ws_parts(a.B, a.H, a.N);
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  float* k_hi = reinterpret_cast<float*>(ws);
  float* k_lo = reinterpret_cast<float*>(ws + w.k_bytes);
  float* vt_hi = reinterpret_cast<float*>(ws + 2 * w.k_bytes);
  __nv_bfloat16* vt_b = reinterpret_cast<__nv_bfloat16*>(ws + 2 * w.k_bytes + w.vt_bytes);
  __nv_bfloat16* vt_lo_b =
      reinterpret_cast<__nv_bfloat16*>(ws + 2 * w.k_bytes + w.vt_bytes + w.vt_bytes / 2);
  CUtensorMap maps[5];
  CUresult r = make_map(&maps[0], k_hi, kD, (cuuint64_t)a.N, BH, 4);
  if (r == CUDA_SUCCESS) r = make_map(&maps[1], k_lo, kD, (cuuint64_t)a.N, BH, 4);
  if (r == CUDA_SUCCESS) r = make_map(&maps[2], vt_hi, (cuuint64_t)w.Np, kD, BH, 4);
  if (r == CUDA_SUCCESS) r = make_map(&maps[3], vt_b, (cuuint64_t)w.Np, kD, BH, 2);
  if (r == CUDA_SUCCESS) r = make_map(&maps[4], vt_lo_b, (cuuint64_t)w.Np, kD, BH, 2);
  if (r != CUDA_SUCCESS) {
    attn_set_error("attn_fwd_tf32x3: cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return cudaErrorInvalidValue;
  }
  tf32x3_split_kernel<<<dim3((unsigned)(w.Np / 64), (unsigned)(BH < 65535 ? BH : 65535)), 256,
                        0, s>>>(a.k, a.v, k_hi, k_lo, vt_hi, vt_b, vt_lo_b, a.N, w.Np, BH);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const float scale_log2 = a.scale * 1.4426950408889634f;
  return a.causal ? launch_t<true>(a, maps, scale_log2, s)
                  : launch_t<false>(a, maps, scale_log2, s);
}
