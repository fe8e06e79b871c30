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
//     columns [0,256) and RoPE columns [512,544), rank 1 owns [256,512) and
//     [544,576) (18 S MMAs each per step).  Each CTA TMA-loads only its own
//     columns of every cached row (HBM is read once) and computes a partial S
//     over them for all 128 heads with its share of q held in TMEM.
//   * The softmax of each head runs on one CTA only: rank r owns heads
//     64 r .. 64 r + 63.  A CTA pushes its partial S of the peer's heads into
//     the peer's shared memory with st.async (two 32-token messages per step,
//     arrival counted in bytes on the peer's mbarrier), adds the peer's
//     partial of its own heads to its own, runs their online softmax, writes
//     their bf16 P rows into a shared-memory P tile and bulk-copies those rows
//     into the peer's tile, with each head's rescale factor.  Both CTAs then
//     accumulate their 256 columns of O = P V in TMEM with P from shared
//     memory (V is the same shared-memory bytes as K), after applying the
//     peer's factors to their O rows of the peer's heads.
//   * Each 64-token page is one step (S MMAs with N=64) through a 4-stage TMA
//     ring of the CTA's c_kv atoms and its 32 RoPE columns; the block table is
//     read on the device and bounds-checked.  Two S buffers in TMEM; since P
//     lives in shared memory, an S buffer is free as soon as it has been
//     read, and S and PV are issued by two threads.  Warps 0-7: softmax of the
//     own heads or service of the peer's heads, by TMEM lane quarter, the two
//     step parities in ping-pong; 8 TMA producer; 9 S-MMA issuer; 10 PV-MMA
//     issuer.  Each PV commit is multicast to both CTAs: a P slot is reused
//     once both CTAs' PVs of the step are done.
//   * Work is a list of page ranges ("chunks") of the flat page order, one
//     chunk per cluster at a time (persistent).  The device planner either
//     gives each sequence its own chunk (no partials) or cuts the flat order
//     into equal chunks, moving cuts to nearby sequence starts; a sequence cut
//     by a chunk edge writes partials (O / l as bf16 rows, the LSE in fp32)
//     that a small combine kernel merges.
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
constexpr int kStep = 64;                 // tokens per MMA step (one page)
constexpr int kOwn = kHq / 2;             // heads whose softmax runs on each CTA
// Warps 0-7 compute (warp w: TMEM lane quarter w % 4, the steps of parity
// w / 4; the softmax for this CTA's 64 heads, or the partial-S sends and O
// upkeep for the peer's 64), 8 TMA producer, 9 S-MMA issuer, 10 PV-MMA issuer.
constexpr int kThreads = 352;
constexpr int kKAtomBytes = kStep * 128;  // 64 tokens x 64 bf16
constexpr int kStageBytes = 4 * kKAtomBytes;  // the CTA's 4 c_kv atoms (K and V): 32 KB
constexpr int kStages = 4;
// The 64 RoPE columns are split between the ranks, 32 each (64-byte rows,
// 64-byte swizzle).  Each stage has a RoPE slot of its own beside its c_kv
// atoms, loaded and released with the stage.
constexpr int kRopeSlots = kStages;
constexpr int kRopeCols = 32;                       // RoPE columns per CTA
constexpr int kRopeRowBytes = kRopeCols * 2;        // 64 B
constexpr int kQropeBytes = kHq * kRopeRowBytes;    // q's RoPE half: 8 KB
constexpr int kKropeBytes = kStep * kRopeRowBytes;  // a step's k_rope half: 4 KB
constexpr int kSBufs = 2;                 // TMEM S buffers (64 columns each)
static_assert((kStages & (kStages - 1)) == 0 && (kSBufs & (kSBufs - 1)) == 0 &&
                  (kRopeSlots & (kRopeSlots - 1)) == 0,
              "ring positions are taken with masks");
// A partial-S message: one 32-token half of a step for the 64 heads of the
// receiving CTA, [token quad][head][4 tokens] fp32: 16 B per head and quad, so
// one warp store covers 512 contiguous bytes (contiguous remote stores move
// about twice the bytes per clock of row-scattered ones) and each head's
// reads are conflict-free.
constexpr int kXQuadBytes = kOwn * 16;                 // 1 KB
constexpr int kXHalf = 32;                             // tokens per message
constexpr int kXMsgBytes = (kXHalf / 4) * kXQuadBytes;  // 8 KB
constexpr int kXSlots = 2 * (kStep / kXHalf);           // two steps x two halves
// P of one step in shared memory (the A operand of the PV MMAs): two K-major
// atoms of 32 tokens (64-byte rows, 64-byte swizzle) over the 128 head rows.
// A warp's 32 rows of one atom are 2 KB contiguous, which is what it copies
// to the peer.
constexpr int kPAtomBytes = kHq * 64;         // 8 KB
constexpr int kPSlotBytes = 2 * kPAtomBytes;  // 16 KB
constexpr int kPSlots = 2;
constexpr int kPWarpBytes = 32 * 64;          // 2 KB
// per step each CTA receives the P rows of the peer's 64 heads and their
// rescale factors; per segment their final row sums
constexpr uint32_t kXpBytes = 4 * kPWarpBytes + kOwn * 4;
constexpr uint32_t kLfinBytes = kOwn * 4;
constexpr float kRescaleThreshold = 8.0f;

constexpr int kQropeOff = 0;             // q's RoPE half (A of 2 S MMAs)
constexpr int kRopeOff = kQropeOff + kQropeBytes;  // the stages' k_rope slots
constexpr int kStageOff = kRopeOff + kRopeSlots * kKropeBytes;
static_assert(kStageOff % 1024 == 0, "swizzled stages start on 1024-byte boundaries");
constexpr int kXOff = kStageOff + kStages * kStageBytes;
constexpr int kPOff = kXOff + kXSlots * kXMsgBytes;
static_assert(kPOff % 1024 == 0, "P atoms start on swizzle-pattern boundaries");
constexpr int kAlphaOff = kPOff + kPSlots * kPSlotBytes;  // [P slot][64] factors from the peer
constexpr int kLfinOff = kAlphaOff + kPSlots * kOwn * 4;   // [segment parity][64] from the peer
constexpr int kMpubOff = kLfinOff + 2 * kOwn * 4;          // [step parity][64] running maxima
constexpr int kLpartOff = kMpubOff + 2 * kOwn * 4;         // [segment parity][step parity][l | m]
constexpr int kBarOff = kLpartOff + 2 * 2 * kOwn * 8;
// barriers: kv_full[S], kv_free[S], s_full[2], s_read[2], x_full[4], x_read[2],
// p_full[2], xp_full[2], lfin_full[2], m_ready[2], kv_empty[S], q_full, q_free,
// o_free, seg_done, drain_s, drain_pv
constexpr int kNumBars = 3 * kStages + 3 * kSBufs + kXSlots + 4 * kPSlots + 6;
constexpr int kMiscOff = (kBarOff + kNumBars * 8 + 15) & ~15;
constexpr int kSmemBytes = kMiscOff + 16 + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;     // 256 columns
constexpr uint32_t kColQ = 256;   // 128 columns: q's four c_kv atoms (bf16 pairs)
constexpr uint32_t kColS = 384;   // 2 x 64 columns

// ---- workspace layout -------------------------------------------------------
struct WsLayout {
  size_t header, prefix, bounds, cstart, clist, plse, po, total;
  int max_chunks;
};

__host__ __device__ constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ constexpr WsLayout ws_layout(int B, int max_chunks) {
  WsLayout w{};
  w.max_chunks = max_chunks;
  w.header = 0;
  w.prefix = 64;
  w.bounds = align_up(w.prefix + sizeof(int) * (size_t)(B + 1), 16);
  w.cstart = align_up(w.bounds + sizeof(int) * (size_t)(max_chunks + 1), 16);
  w.clist = align_up(w.cstart + sizeof(int) * (size_t)max_chunks, 16);
  w.plse = align_up(w.clist + sizeof(int4) * (size_t)B, 256);
  w.po = align_up(w.plse + sizeof(float) * (size_t)(2 * max_chunks) * kHq, 256);
  w.total = align_up(w.po + sizeof(__nv_bfloat16) * (size_t)(2 * max_chunks) * kHq * kDv, 256);
  return w;
}

inline int max_chunks_for(int B, int max_blocks, int num_sms, int pps) {
  if (pps > 0) {
    const long long total = (long long)B * max_blocks;
    return (int)((total + pps - 1) / pps);
  }
  return num_sms / 2;  // per-sequence chunks only when B <= clusters
}

__device__ __forceinline__ int find_range(const int* __restrict__ edges, int n, int x) {
  // largest i in [0, n) with edges[i] <= x < edges[i+1] (edges non-decreasing)
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (edges[mid + 1] <= x) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// ---- plan -------------------------------------------------------------------
// One CTA.  Validates lengths, writes the exclusive page prefix, then the
// chunk edges, by a time model: per-sequence chunks (no partials); with fewer
// sequences than clusters, each sequence cut into near-equal chunks of its
// own; else ceil(T / clusters) pages per chunk with each cut moved to a
// sequence start within 1/8 chunk; or a fixed split length when one is forced.
__global__ void __launch_bounds__(1024) mla_plan_kernel(const int32_t* __restrict__ seqlens,
                                                        int B, int max_blocks, int clusters,
                                                        int pps_override, int* __restrict__ hdr,
                                                        int* __restrict__ prefix,
                                                        int* __restrict__ bounds,
                                                        int* __restrict__ cstart,
                                                        int4* __restrict__ clist, int* err) {
  __shared__ int warp_sums[32];
  __shared__ int warp_max[32];
  __shared__ int carry, maxn_s, nchunks_s, pps_s, mode_s;
  // launched as a programmatic dependent of whatever precedes it on the
  // stream: wait for it before reading the lengths, then let the decode
  // kernel set itself up while this plan runs
  grid_dependency_wait();
  grid_launch_dependents();
  if (threadIdx.x == 0) { carry = 0; maxn_s = 0; }
  __syncthreads();
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int n = 0;
    if (b < B) {
      const int L = seqlens[b];
      if (L < 0 || L > max_blocks * kPage) record_error(err, ATTN_ERR_BAD_SEQLEN, 0, b);
      else n = (L + kPage - 1) / kPage;
    }
    int x = n, mx = n;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    }
    if (lane == 31) warp_sums[wid] = x;
    if (lane == 0) warp_max[wid] = mx;
    __syncthreads();
    if (wid == 0) {
      int w = warp_sums[lane];
      int m = warp_max[lane];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, off);
        if (lane >= off) w += y;
        m = max(m, __shfl_xor_sync(0xffffffffu, m, off));
      }
      warp_sums[lane] = w;
      if (lane == 0) maxn_s = max(maxn_s, m);
    }
    __syncthreads();
    const int incl = x + (wid > 0 ? warp_sums[wid - 1] : 0) + carry;
    if (b < B) prefix[b] = incl - n;
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) carry = incl;
    __syncthreads();
  }
  // Fewer than half as many sequences as clusters (at most 64): each sequence
  // may be cut into ceil(n_b / L) near-equal chunks of its own, L the shortest
  // chunk length whose chunk count fits the clusters.  Warp 0 finds L with
  // one sequence pair per lane; `cut` counts the chunks of cut sequences.
  __shared__ int len3_s, n3_s, cut3_s;
  if (threadIdx.x == 0) prefix[B] = carry;
  __syncthreads();
  if (wid == 0) {
    const bool try3 = pps_override <= 0 && 2 * B <= clusters && B <= 64 && carry > 0;
    const int n0 = (try3 && lane < B) ? prefix[lane + 1] - prefix[lane] : 0;
    const int n1 = (try3 && lane + 32 < B) ? prefix[lane + 33] - prefix[lane + 32] : 0;
    auto warp_sum = [&](int v) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      return v;
    };
    int len = 0, total = 0, cut = 0;
    if (try3) {
      int lo = max(1, (carry + clusters - 1) / clusters), hi = max(lo, maxn_s);
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        const int t = warp_sum((n0 + mid - 1) / mid + (n1 + mid - 1) / mid);
        if (t <= clusters) hi = mid;
        else lo = mid + 1;
      }
      len = lo;
      const int c0 = (n0 + len - 1) / len, c1 = (n1 + len - 1) / len;
      total = warp_sum(c0 + c1);
      cut = warp_sum((c0 > 1 ? c0 : 0) + (c1 > 1 ? c1 : 0));
    }
    if (lane == 0) {
      len3_s = len;
      n3_s = total;
      cut3_s = cut;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const int T = carry;
    int mode, pps, nchunks;
    if (pps_override > 0) {
      mode = 0;
      pps = pps_override;
      nchunks = (T + pps - 1) / pps;
    } else {
      pps = max(1, (T + clusters - 1) / max(clusters, 1));
      // time model: per-cluster pages (tensor-bound) vs bytes (HBM-bound),
      // split partials cost 2 x 128 KB of traffic each (bf16 rows)
      const float page_us = 0.65f, bytes_per_us = 6.5e6f;
      const float kv = (float)T * kPage * 1152.f;
      const int n_a = (T + pps - 1) / pps;
      const float est_a = fmaxf(pps * page_us, (kv + 2.f * n_a * 2.f * 131072.f) / bytes_per_us);
      const float est_b = fmaxf(maxn_s * page_us, kv / bytes_per_us);
      // fewer sequences than clusters: each sequence in ceil(n_b / L) chunks
      // of its own (no chunk spans two sequences), L the shortest chunk
      // length whose chunk count fits the clusters; each chunk of a cut
      // sequence writes one partial (128 KB written, then read)
      const int len_c = len3_s, n_c = n3_s;
      const float est_c =
          len_c > 0 ? fmaxf(len_c * page_us, (kv + 2.f * cut3_s * 131072.f) / bytes_per_us)
                    : 3.4e38f;
      if (B <= clusters && est_b <= est_a && est_b <= est_c) {
        mode = 1;
        nchunks = B;
      } else if (est_c <= est_a) {
        mode = 3;  // the chunk edges are written by warp 0 below
        nchunks = n_c;
        pps = len_c;
      } else {
        mode = 2;
        nchunks = n_a;
      }
    }
    mode_s = mode;
    pps_s = pps;
    nchunks_s = nchunks;
    hdr[0] = T;
    hdr[1] = nchunks;
    hdr[2] = pps;
    hdr[3] = mode;
  }
  __syncthreads();
  const int T = carry, mode = mode_s, pps = pps_s, nchunks = nchunks_s;
  if (mode == 3 && wid == 0) {
    // lane l writes the chunks of sequences l and l + 32, after a scan of
    // the chunk counts gives each sequence its first chunk index
    int first = 0;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int b = lane + 32 * half;
      const int n = (b < B) ? prefix[b + 1] - prefix[b] : 0;
      const int c = (n + pps - 1) / pps;
      int x = c;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
      }
      const int k0 = first + x - c;
      for (int j = 0; j < c; ++j) {
        bounds[k0 + j] = prefix[b] + (int)((long long)j * n / c);
        cstart[k0 + j] = b;
      }
      first += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) bounds[nchunks] = T;
  }
  for (int k = threadIdx.x; k <= nchunks && mode != 3; k += blockDim.x) {  // 3: done above
    int x;
    if (mode == 1) {
      x = prefix[k];
    } else {
      x = min(k * pps, T);
      if (mode == 2 && k > 0 && k < nchunks) {
        const int b = find_range(prefix, B, x);
        const int s0 = prefix[b], s1 = prefix[b + 1];
        const int tol = pps / 8;
        if (x - s0 <= s1 - x) {
          if (x - s0 <= tol) x = s0;
        } else if (s1 - x <= tol) {
          x = s1;
        }
      }
    }
    bounds[k] = x;
    // the sequence holding the chunk's first page (B past the last page):
    // the decode kernel starts each chunk from it without a search
    if (k < nchunks) cstart[k] = (x < T) ? find_range(prefix, B, x) : B;
  }
  // The sequences the combine kernel has to finish, in order: empty ones
  // (O = 0, LSE = -inf) and those cut by a chunk edge (partials to merge).
  // Every other sequence is written whole by the decode kernel.
  __syncthreads();  // every chunk edge is in place
  __shared__ int ccarry;
  if (threadIdx.x == 0) ccarry = 0;
  __syncthreads();
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int f = 0, k0 = -1, k1 = -1;
    if (b < B) {
      const int pb = prefix[b], pe = prefix[b + 1];
      if (pe == pb) {
        f = 1;
      } else {
        k0 = find_range(bounds, nchunks, pb);
        k1 = find_range(bounds, nchunks, pe - 1);
        f = k0 != k1;
      }
    }
    int x = f;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) warp_sums[wid] = x;
    __syncthreads();
    if (wid == 0) {
      int w = warp_sums[lane];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, off);
        if (lane >= off) w += y;
      }
      warp_sums[lane] = w;
    }
    __syncthreads();
    const int incl = x + (wid > 0 ? warp_sums[wid - 1] : 0) + ccarry;
    if (f) {
      // {sequence, first chunk, last chunk, slot of the first chunk's partial}
      // (a chunk's second segment writes slot 2k + 1); k0 = -1: empty sequence
      const int first_slot = (k0 >= 0) ? (bounds[k0] != prefix[b] ? 2 * k0 + 1 : 2 * k0) : -1;
      clist[incl - 1] = make_int4(b, k0, k1, first_slot);
    }
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) ccarry = incl;
    __syncthreads();
  }
  if (threadIdx.x == 0) hdr[4] = ccarry;
}

// ---- decode -----------------------------------------------------------------
struct Seg {
  int b, p0, p1;  // sequence and its page range [p0, p1)
  int slot;       // partial slot, or -1 when the segment is the whole sequence
};

// Enumerates the sequence segments of chunk k in order.
struct ChunkIter {
  const int* prefix;
  int B, k, start, end, first_page, b;
  __device__ void init(const int* pf, const int* bounds, const int* cstart, int B_, int k_) {
    prefix = pf; B = B_; k = k_;
    start = bounds[k];
    end = bounds[k + 1];
    first_page = start;
    b = (start < end) ? cstart[k] : B;
  }
  __device__ bool next(Seg& s) {
    if (start >= end || b >= B) return false;
    const int seg_end = min(end, prefix[b + 1]);
    s.b = b;
    s.p0 = start - prefix[b];
    s.p1 = seg_end - prefix[b];
    const int npages = prefix[b + 1] - prefix[b];
    const bool whole = (s.p0 == 0 && s.p1 == npages);
    const bool first = (start == first_page);
    s.slot = whole ? -1 : (first ? 2 * k : 2 * k + 1);
    start = seg_end;
    ++b;
    while (b < B && prefix[b + 1] <= start) ++b;
    return true;
  }
};

__device__ __forceinline__ int seg_steps(int p0, int p1, int L) {
  const int t0 = p0 * kPage, t_end = min(p1 * kPage, L);
  return (t_end - t0 + kStep - 1) / kStep;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tmKV,
                      const __grid_constant__ CUtensorMap tmRope,
                      const __nv_bfloat16* __restrict__ q,
                      const int32_t* __restrict__ block_table,
                      const int32_t* __restrict__ seqlens, __nv_bfloat16* __restrict__ o,
                      float* __restrict__ lse, const int* __restrict__ hdr,
                      const int* __restrict__ prefix, const int* __restrict__ bounds,
                      const int* __restrict__ cstart,
                      float* __restrict__ part_lse, __nv_bfloat16* __restrict__ part_o, int B,
                      int max_blocks, int num_blocks, float scale_log2, int* err,
                      int debug_skip_step) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);

  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int cluster = blockIdx.x >> 1;
  const int nclusters = gridDim.x >> 1;

  // columns owned by this CTA: four 64-column c_kv atoms of the 576-wide row
  // and one half of the RoPE columns
  auto atom_col = [&](int a) -> int { return (int)rank * 256 + a * 64; };
  const int rope_col = 512 + (int)rank * kRopeCols;

  const uint32_t sQrope = base + kQropeOff;
  const uint32_t sRope = base + kRopeOff;
  const uint32_t sStage = base + kStageOff;
  const uint32_t sX = base + kXOff;
  const uint32_t sP = base + kPOff;
  const uint32_t bar0 = base + kBarOff;
  constexpr int kBarX = 2 * kStages + 2 * kSBufs;
  constexpr int kBarP = kBarX + kXSlots + kSBufs;
  auto bar_kv_full = [&](int s) { return bar0 + 8u * s; };
  // kv_free(s) completes when the PV of the stage's step is done on BOTH CTAs
  // (that PV commit is multicast): it frees the P slot of the step two later.
  auto bar_kv_free = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto bar_s_full = [&](int b) { return bar0 + 8u * (2 * kStages + b); };
  auto bar_s_read = [&](int b) { return bar0 + 8u * (2 * kStages + kSBufs + b); };
  auto bar_x_full = [&](int x) { return bar0 + 8u * (kBarX + x); };
  auto bar_x_read = [&](int x) { return bar0 + 8u * (kBarX + kXSlots + x); };
  auto bar_p_full = [&](int b) { return bar0 + 8u * (kBarP + b); };
  auto bar_xp_full = [&](int b) { return bar0 + 8u * (kBarP + kPSlots + b); };
  auto bar_lfin_full = [&](int b) { return bar0 + 8u * (kBarP + 2 * kPSlots + b); };
  // m_ready(b): the softmax warps of a step of parity b have published the
  // running max after it (the next step's warps need it)
  auto bar_m_ready = [&](int b) { return bar0 + 8u * (kBarP + 3 * kPSlots + b); };
  // kv_empty(s): the PV of the stage's step is done on this CTA: the stage is
  // free for the producer, and the O rescales and the epilogue learn from it
  // that a PV is done.
  auto bar_kv_empty = [&](int s) { return bar0 + 8u * (kBarP + 4 * kPSlots + s); };
  const uint32_t bar_q_full = bar0 + 8u * (kBarP + 4 * kPSlots + kStages);
  const uint32_t bar_q_free = bar_q_full + 8;
  const uint32_t bar_o_free = bar_q_full + 16;
  const uint32_t bar_seg_done = bar_q_full + 24;
  const uint32_t bar_drain_s = bar_q_full + 32;
  const uint32_t bar_drain_pv = bar_q_full + 40;
  static_assert(kBarP + 4 * kPSlots + kStages + 6 == kNumBars, "barrier count");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kMiscOff + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_kv_full(s), 1);
      mbar_init(bar_kv_free(s), 2);
      mbar_init(bar_kv_empty(s), 1);
    }
    for (int b = 0; b < kSBufs; ++b) {
      mbar_init(bar_s_full(b), 1);
      mbar_init(bar_s_read(b), 4);  // the four compute warps of the step's parity
    }
    for (int x = 0; x < kXSlots; ++x) mbar_init(bar_x_full(x), 1);
    for (int b = 0; b < kSBufs; ++b) mbar_init(bar_x_read(b), 2);  // the step's softmax warps
    for (int b = 0; b < kPSlots; ++b) {
      mbar_init(bar_p_full(b), 4);
      mbar_init(bar_xp_full(b), 1);
      mbar_init(bar_lfin_full(b), 1);
      mbar_init(bar_m_ready(b), 2);
    }
    mbar_init(bar_q_full, 8);
    mbar_init(bar_q_free, 1);
    mbar_init(bar_o_free, 8);
    mbar_init(bar_seg_done, 4);  // the four softmax warps
    mbar_init(bar_drain_s, 1);
    mbar_init(bar_drain_pv, 1);
    *abort_flag = 0;
    fence_mbar_init();
    // arm the barriers that count the peer's bytes (re-armed after each use)
    for (int x = 0; x < kXSlots; ++x) mbar_arrive_expect_tx(bar_x_full(x), kXMsgBytes);
    for (int b = 0; b < kPSlots; ++b) {
      mbar_arrive_expect_tx(bar_xp_full(b), kXpBytes);
      mbar_arrive_expect_tx(bar_lfin_full(b), kLfinBytes);
    }
    prefetch_tmap(&tmKV);
    prefetch_tmap(&tmRope);
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers are initialised before any remote access
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  // The set-up above overlaps the plan kernel; its chunk list is read only
  // now.  A cluster without a chunk runs no role loop and goes to teardown.
  grid_dependency_wait();
  grid_launch_dependents();  // the combine kernel may be scheduled
  const int nchunks = hdr[1];

  if (warp == 8) {
    // ================= producer: paged K/V (own columns) =================
    if (lane == 0) {
      const uint64_t pol_kv = policy_evict_first();  // every cached row is read once
      // test hook: rank 1 of every cluster never loads this step
      const int skip_step = rank == 1 ? debug_skip_step : -1;
      int g = 0, issued = 0, skipped = -1;
      bool ok = true;
      for (int k = cluster; k < nchunks && ok; k += nclusters) {
        ChunkIter it;
        it.init(prefix, bounds, cstart, B, k);
        Seg s;
        while (ok && it.next(s)) {
          const int L = seqlens[s.b];
          const int t_end = min(s.p1 * kPage, L);
          for (int t = s.p0 * kPage; t < t_end; t += kStep, ++g) {
            const int slot = g % kStages, use = g / kStages;
            // the page's table entry is read while the stage is still in use
            int blk = block_table[(size_t)s.b * max_blocks + t / kPage];
            if (use > 0) {
              ok = mbar_wait(bar_kv_empty(slot), (use - 1) & 1, abort_flag, err, kSiteKvEmpty, g);
              if (!ok) break;
            }
            if (g == skip_step) {
              skipped = g;
              issued = g + 1;
              continue;
            }
            if (blk < 0 || blk >= num_blocks) {
              record_error(err, ATTN_ERR_BAD_BLOCK_TABLE, s.b, t / kPage);
              blk = 0;  // never read outside the pool
            }
            const int row = blk * kPage + (t % kPage);
            const uint32_t dst = sStage + slot * kStageBytes;
            // the c_kv atoms and the RoPE half into the stage, all counted on
            // the stage's full barrier
            mbar_arrive_expect_tx(bar_kv_full(slot), 4 * kKAtomBytes + kKropeBytes);
            for (int a = 0; a < 4; ++a)
              tma_load_2d_hint(dst + a * kKAtomBytes, &tmKV, bar_kv_full(slot), atom_col(a), row,
                               pol_kv);
            tma_load_2d_hint(sRope + slot * kKropeBytes, &tmRope, bar_kv_full(slot), rope_col, row,
                             pol_kv);
            issued = g + 1;
          }
        }
      }
      if (!ok) {
        const int first = issued > kStages ? issued - kStages : 0;
        for (int gg = first; gg < issued; ++gg) {
          if (gg == skipped) continue;
          volatile int never = 0;
          mbar_wait(bar_kv_full(gg % kStages), (gg / kStages) & 1, &never, nullptr, kSiteDrain, gg);
        }
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ================= S issuer: partial S over this CTA's columns ==========
    // S of a step needs only its stage and a free S buffer (P lives in shared
    // memory), so this thread runs ahead of the PVs.
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_bf16(kHq, kStep, false, false);  // N = 64 tokens
      const uint32_t tQ = tbase + kColQ;
      // Descriptors are built once; per MMA only the start address moves
      // (the 14-bit address field never carries into the other fields).
      const uint64_t kdesc0 = sdesc_sw128(sStage, 16, 1024);
      const uint64_t qrdesc = sdesc_sw64(sQrope, 512);
      const uint64_t kropedesc0 = sdesc_sw64(sRope, 512);
      int g = 0, seg_i = 0;
      bool ok = true;
      for (int k = cluster; k < nchunks && ok; k += nclusters) {
        ChunkIter it;
        it.init(prefix, bounds, cstart, B, k);
        Seg s;
        while (ok && it.next(s)) {
          const int n = seg_steps(s.p0, s.p1, seqlens[s.b]);
          ok = mbar_wait(bar_q_full, seg_i & 1, abort_flag, err, kSiteQFull, seg_i);
          if (!ok) break;
          tc_fence_after();
          for (int i = 0; i < n; ++i) {
            const uint32_t u = (uint32_t)(g + i);
            const uint32_t sb = u & (kSBufs - 1);
            const uint32_t slot = u & (kStages - 1);
            // every compute warp has read the buffer's previous S
            if (u >= (uint32_t)kSBufs) {
              ok = mbar_wait(bar_s_read(sb), ((u - kSBufs) / kSBufs) & 1u, abort_flag, err,
                             kSiteXfree, (int)u);
              if (!ok) break;
            }
            ok = mbar_wait(bar_kv_full(slot), (u / kStages) & 1u, abort_flag, err, kSiteKvFull,
                           (int)u);
            if (!ok) break;
            tc_fence_after();
            const uint64_t kd = kdesc0 + (uint64_t)((slot * kStageBytes) >> 4);
            const uint32_t tS = tbase + kColS + sb * 64;
            // c_kv atoms: q from TMEM; the RoPE half: q from shared memory
#pragma unroll
            for (int a = 0; a < 4; ++a) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_ts(tS, tQ + a * 32 + kk * 8,
                       kd + (uint64_t)((a * kKAtomBytes + kk * 32) >> 4), kIdescS,
                       (a | kk) != 0);
            }
            const uint64_t rd = kropedesc0 + (uint64_t)((slot * kKropeBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < kRopeCols / 16; ++kk)
              mma_ss(tS, qrdesc + (uint64_t)((kk * 32) >> 4), rd + (uint64_t)((kk * 32) >> 4),
                     kIdescS, 1u);
            tc_commit(bar_s_full(sb));
          }
          if (!ok) break;
          tc_commit(bar_q_free);  // every reader of this segment's q issued
          g += n;
          ++seg_i;
        }
      }
      tc_commit(bar_drain_s);
      volatile int never = 0;
      mbar_wait(bar_drain_s, 0, &never, nullptr, kSiteDrain, -2);
    }
    __syncwarp();
  } else if (warp == 10) {
    // ================= PV issuer: O[:, own columns] += P V ==================
    if (lane == 0) {
      constexpr uint32_t kIdescPV = idesc_bf16(kHq, 256, false, true);
      const uint32_t tO = tbase + kColO;
      const uint64_t pdesc0 = sdesc_sw64(sP, 512);
      const uint64_t vdesc0 = sdesc_sw128(sStage, kKAtomBytes, 1024);
      int g = 0, seg_i = 0;
      bool ok = true;
      for (int k = cluster; k < nchunks && ok; k += nclusters) {
        ChunkIter it;
        it.init(prefix, bounds, cstart, B, k);
        Seg s;
        while (ok && it.next(s)) {
          const int n = seg_steps(s.p0, s.p1, seqlens[s.b]);
          if (seg_i > 0) {  // the previous segment's epilogue has read O
            ok = mbar_wait(bar_o_free, (seg_i - 1) & 1, abort_flag, err, kSitePvDone, seg_i);
            if (!ok) break;
          }
          for (int i = 0; i < n; ++i) {
            const uint32_t u = (uint32_t)(g + i);
            const uint32_t pb = u & (kPSlots - 1);
            const uint32_t slot = u & (kStages - 1);
            ok = mbar_wait(bar_p_full(pb), (u / kPSlots) & 1u, abort_flag, err, kSitePFull,
                           (int)u);
            if (!ok) break;
            tc_fence_after();
            const uint64_t pd = pdesc0 + (uint64_t)((pb * kPSlotBytes) >> 4);
            const uint64_t vd = vdesc0 + (uint64_t)((slot * kStageBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < kStep / 16; ++kk)
              mma_ss(tO, pd + (uint64_t)(((kk >> 1) * kPAtomBytes + (kk & 1) * 32) >> 4),
                     vd + (uint64_t)((kk * 16 * 128) >> 4), kIdescPV, (i | kk) != 0);
            tc_commit(bar_kv_empty(slot));
            tc_commit_mc(bar_kv_free(slot), 0x3);
          }
          if (!ok) break;
          g += n;
          ++seg_i;
        }
      }
      tc_commit(bar_drain_pv);
      volatile int never = 0;
      mbar_wait(bar_drain_pv, 0, &never, nullptr, kSiteDrain, -3);
    }
    __syncwarp();
  } else {
    // ================= compute warps 0-7 =================
    // Warp w covers TMEM lanes (heads) 32 (w % 4) .. + 31 and the steps of
    // parity w / 4.  Heads 64 rank .. + 63 are this CTA's own: their warps run
    // the softmax of whole 64-token rows, the two parities in ping-pong (a warp
    // has two steps' time for one, so one warp's waits overlap the other's
    // work).  The other warps serve the peer's heads: they send this CTA's
    // partial S of those heads and keep those heads' O rows (this CTA's
    // columns) in step with the peer's softmax.  In the epilogue warp w writes
    // O columns 128 (w / 4) .. + 127 of its rows.
    const int sub = warp & 3, par = warp >> 2;
    const bool own = (sub >> 1) == (int)rank;
    const int h = sub * 32 + lane;       // head == TMEM lane
    const int j = h & (kOwn - 1);        // its index among its owner's 64 heads
    const uint32_t lane_off = (uint32_t)(sub * 32) << 16;
    const uint32_t tO = tbase + lane_off + kColO;
    const uint32_t tQ = tbase + lane_off + kColQ;
    const uint32_t tS = tbase + lane_off + kColS;
    const bool first_of_pair = (sub & 1) == 0;  // one warp per (role, parity) arms barriers
    const float* lfin = reinterpret_cast<const float*>(smem + kLfinOff);
    const float* alpha_in = reinterpret_cast<const float*>(smem + kAlphaOff);
    float* mpub = reinterpret_cast<float*>(smem + kMpubOff);
    float* lpart = reinterpret_cast<float*>(smem + kLpartOff);
    const uint32_t peer_x = mapa_shared(sX + j * 16, peer);
    const uint32_t peer_x_full0 = mapa_shared(bar_x_full(0), peer);
    const uint32_t peer_alpha = mapa_shared(base + kAlphaOff + j * 4, peer);
    const uint32_t peer_lfin = mapa_shared(base + kLfinOff + j * 4, peer);
    const uint32_t peer_xp_full0 = mapa_shared(bar_xp_full(0), peer);
    const uint32_t peer_lfin_full0 = mapa_shared(bar_lfin_full(0), peer);
    const uint32_t peer_p = mapa_shared(sP, peer);
    constexpr float kLn2 = 0.69314718055994530942f;
    int g = 0, seg_i = 0;
    bool ok = true;
    // the previous segment, whose epilogue runs once the next q is in place
    int prev_b = -1, prev_slot = -1, prev_seg = 0, prev_last = 0;
    float prev_m = 0.f, prev_l = 0.f;

    // this warp's rows of O (all 256 of this CTA's columns) times a
    auto rescale_o = [&](float a) {
#pragma unroll 1
      for (int c = 0; c < 256; c += 32) {
        float ov[32];
        tmem_ld32(tO + c, ov);
        uint32_t ou[32];
#pragma unroll
        for (int u = 0; u < 32; ++u) ou[u] = __float_as_uint(ov[u] * a);
        tmem_st32(tO + c, ou);
      }
      tmem_st_wait();
    };

    // O / l of this warp's rows and columns -> bf16, into O (whole sequence)
    // or into the segment's partial slot; the LSE of its own heads (fp32).  The peer's heads take the row
    // sums the peer sent.
    auto epilogue = [&]() -> bool {
      float lv = prev_l;
      if (!own) {
        const int ls = prev_seg & 1;
        const bool w = mbar_wait<true>(bar_lfin_full(ls), (prev_seg >> 1) & 1, abort_flag, err,
                                       kSiteXchg, prev_seg);
        if (!__all_sync(0xffffffffu, w)) return false;
        lv = lfin[ls * kOwn + j];
        if (first_of_pair && par == 0 && lane == 0)
          mbar_arrive_expect_tx(bar_lfin_full(ls), kLfinBytes);  // for two segments on
      }
      const float inv_l = (lv > 0.f) ? 1.0f / lv : 0.f;
      const size_t orow = (size_t)prev_b * kHq + h;
      const int col0 = (int)rank * 256 + par * 128;
#pragma unroll 1
      for (int c = 0; c < 128; c += 32) {
        float ov[32];
        tmem_ld32(tO + par * 128 + c, ov);
        __nv_bfloat16* dst =
            (prev_slot < 0 ? o + orow * kDv : part_o + ((size_t)prev_slot * kHq + h) * kDv) +
            col0 + c;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint4 w;
          w.x = pack_bf16x2(ov[q4 * 8 + 0] * inv_l, ov[q4 * 8 + 1] * inv_l);
          w.y = pack_bf16x2(ov[q4 * 8 + 2] * inv_l, ov[q4 * 8 + 3] * inv_l);
          w.z = pack_bf16x2(ov[q4 * 8 + 4] * inv_l, ov[q4 * 8 + 5] * inv_l);
          w.w = pack_bf16x2(ov[q4 * 8 + 6] * inv_l, ov[q4 * 8 + 7] * inv_l);
          *reinterpret_cast<uint4*>(dst + q4 * 8) = w;
        }
      }
      if (own && par == 0) {
        const float lse_v = (lv > 0.f) ? (prev_m + log2f(lv)) * kLn2 : -INFINITY;
        if (prev_slot < 0) lse[orow] = lse_v;
        else part_lse[(size_t)prev_slot * kHq + h] = lse_v;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_o_free);
      return true;
    };

    for (int k = cluster; k < nchunks && ok; k += nclusters) {
      ChunkIter it;
      it.init(prefix, bounds, cstart, B, k);
      Seg s;
      while (ok && it.next(s)) {
        const int L = seqlens[s.b];
        const int t0 = s.p0 * kPage;
        const int n = seg_steps(s.p0, s.p1, L);
        // ---- this segment's q: this warp's heads, c_kv atoms 2 par and
        //      2 par + 1 -> TMEM (A operand of the S MMAs); the RoPE half ->
        //      shared memory
        if (seg_i > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(bar_q_free, (seg_i - 1) & 1, abort_flag, err,
                                                 kSiteQFull, seg_i));
          if (!ok) break;
        }
        {
          const uint4* qrow = reinterpret_cast<const uint4*>(q + ((size_t)s.b * kHq + h) * kDk);
          uint4 qv[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) qv[c] = __ldg(qrow + atom_col(2 * par) / 8 + c);
          uint4 rv[4];
          if (par == 0) {
#pragma unroll
            for (int c = 0; c < 4; ++c) rv[c] = __ldg(qrow + rope_col / 8 + c);
          }
#pragma unroll
          for (int a = 0; a < 2; ++a) {
            uint32_t w[32];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint4 v = qv[a * 8 + c];
              w[4 * c] = v.x; w[4 * c + 1] = v.y; w[4 * c + 2] = v.z; w[4 * c + 3] = v.w;
            }
            tmem_st32(tQ + (2 * par + a) * 32, w);
          }
          if (par == 0) {
            // 64-byte rows with the 64-byte swizzle: 16-byte chunk c of row r
            // at chunk c ^ ((r >> 1) & 3)
            uint8_t* qr = smem + kQropeOff + h * kRopeRowBytes;
#pragma unroll
            for (int c = 0; c < 4; ++c)
              *reinterpret_cast<uint4*>(qr + ((c ^ ((h >> 1) & 3)) * 16)) = rv[c];
            fence_proxy_async_smem();
          }
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_q_full);
        }
        // the next segment of this chunk: this thread's q lines into L2, so
        // that its load at the segment change does not wait on DRAM
        if (it.start < it.end && it.b < B) {
          const char* nq = reinterpret_cast<const char*>(q + ((size_t)it.b * kHq + h) * kDk);
          asm volatile("prefetch.global.L2 [%0];" ::"l"(nq + atom_col(2 * par) * 2));
          asm volatile("prefetch.global.L2 [%0];" ::"l"(nq + atom_col(2 * par) * 2 + 128));
          if (par == 0) asm volatile("prefetch.global.L2 [%0];" ::"l"(nq + rope_col * 2));
        }
        // ---- the previous segment's epilogue overlaps this segment's first S
        if (prev_b >= 0) {
          ok = __all_sync(0xffffffffu,
                          mbar_wait(bar_kv_empty(prev_last & (kStages - 1)),
                                    (prev_last / kStages) & 1, abort_flag, err, kSitePvDone,
                                    prev_seg));
          if (!ok) break;
          tc_fence_after();
          ok = epilogue();
          if (!ok) break;
          prev_b = -1;
        }
        if (own) {
          // ================= softmax of this CTA's heads =================
          float m_known = -INFINITY;  // the running max this warp's l is relative to
          float l = 0.f;              // this warp's share of the row sum
          for (int i = (par - g) & 1; i < n; i += 2) {
            const int gi = g + i;
            const int b = gi & 1;  // S buffer, message slots and P slot of the step
            const int nvalid = L - (t0 + i * kStep);
            bool w = mbar_wait(bar_s_full(b), (gi >> 1) & 1, abort_flag, err, kSiteSFull, gi);
            if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
            tc_fence_after();
            float t[kStep];
            tmem_ld64(tS + b * 64, t);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_s_read(b));
            // The score is this CTA's partial plus the peer's.  The peer's
            // arrives in two 32-token halves: the first is summed, scaled
            // (log2 units; tokens past the end -inf) and maxed while the
            // second is still on its way.
            float mx0 = -INFINITY, mx1 = -INFINITY;
            bool xok = true;
#pragma unroll
            for (int hx = 0; hx < 2; ++hx) {
              const int xs = b * 2 + hx;
              xok = __all_sync(0xffffffffu, mbar_wait<true>(bar_x_full(xs), (gi >> 1) & 1,
                                                              abort_flag, err, kSiteXchg, gi));
              if (!xok) break;
              const uint8_t* xin = smem + kXOff + xs * kXMsgBytes + j * 16;
#pragma unroll
              for (int c = hx * kXHalf; c < (hx + 1) * kXHalf; c += 4) {
                const float4 pv =
                    *reinterpret_cast<const float4*>(xin + ((c - hx * kXHalf) / 4) * kXQuadBytes);
                fadd2_acc(t[c], t[c + 1], pv.x, pv.y);
                fadd2_acc(t[c + 2], t[c + 3], pv.z, pv.w);
              }
              if (nvalid >= kStep) {
#pragma unroll
                for (int c = hx * kXHalf; c < (hx + 1) * kXHalf; c += 4) {
                  ffma2(t[c], t[c + 1], t[c], t[c + 1], scale_log2, scale_log2, 0.f, 0.f);
                  ffma2(t[c + 2], t[c + 3], t[c + 2], t[c + 3], scale_log2, scale_log2, 0.f, 0.f);
                  mx0 = fmax3(mx0, t[c], t[c + 1]);
                  mx1 = fmax3(mx1, t[c + 2], t[c + 3]);
                }
              } else {
#pragma unroll
                for (int c = hx * kXHalf; c < (hx + 1) * kXHalf; ++c) {
                  t[c] = (c < nvalid) ? t[c] * scale_log2 : -INFINITY;
                  mx0 = fmaxf(mx0, t[c]);
                }
              }
            }
            if (!xok) {
              ok = false;
              break;
            }
            __syncwarp();
            if (lane == 0) {
              mbar_arrive(bar_x_read(b));
              if (first_of_pair) {  // both halves, for step gi + 2
                mbar_arrive_expect_tx(bar_x_full(b * 2), kXMsgBytes);
                mbar_arrive_expect_tx(bar_x_full(b * 2 + 1), kXMsgBytes);
              }
            }
            const float mx = fmaxf(mx0, mx1);
            // the running max after the previous step, published by the warp
            // of the other parity (a segment starts from -inf)
            float m_prev = -INFINITY;
            if (i > 0) {
              const int gp = gi - 1;
              w = mbar_wait(bar_m_ready(gp & 1), (gp >> 1) & 1, abort_flag, err, kSiteXchg, gi);
              if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
              m_prev = mpub[(gp & 1) * kOwn + j];
            }
            // catch up with rescales made at steps of the other parity
            if (m_prev > m_known) {
              l *= fast_exp2(m_known - m_prev);
              m_known = m_prev;
            }
            // lazy rescale: the reference moves only when the row max passes
            // it by more than the threshold (P then stays below 2^threshold)
            const float m_new = fmaxf(m_prev, mx);
            const bool resc = m_new > m_prev + kRescaleThreshold;
            const float alpha = resc ? fast_exp2(m_prev - m_new) : 1.f;  // 0 from -inf
            if (resc) {
              l *= alpha;
              m_known = m_new;
            }
            mpub[b * kOwn + j] = m_known;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_m_ready(b));
            const float nm = (m_known == -INFINITY) ? 0.f : -m_known;
            // O rows of these heads: rescaled once the previous step's PV is
            // done on this CTA
            if (i > 0 && __any_sync(0xffffffffu, resc)) {
              const int gp = gi - 1;
              w = mbar_wait(bar_kv_empty(gp & (kStages - 1)), (gp / kStages) & 1,
                            abort_flag, err, kSitePvDone, gi);
              if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
              tc_fence_after();
              rescale_o(alpha);
            }
            // the step's P slot is free once both CTAs' PV of step gi - 2 is done
            if (gi >= kPSlots) {
              const int gp = gi - kPSlots;
              w = mbar_wait<true>(bar_kv_free(gp & (kStages - 1)), (gp / kStages) & 1,
                                  abort_flag, err, kSiteXfree, gi);
              if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
            }
            // the peer scales its O rows of these heads by the same factor
            st_async_b32(peer_alpha + b * kOwn * 4, __float_as_uint(alpha),
                         peer_xp_full0 + 8u * b);
            // P one 32-token atom at a time; each atom's rows of these heads go
            // to the peer as soon as they are written
            float rr[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) rr[u] = 0.f;
#pragma unroll
            for (int a = 0; a < 2; ++a) {
              uint32_t p[16];
#pragma unroll
              for (int c = 0; c < 32; c += 8) {
                float tv[8], pv[8];
#pragma unroll
                for (int u = 0; u < 8; u += 2)
                  ffma2(tv[u], tv[u + 1], t[a * 32 + c + u], t[a * 32 + c + u + 1], 1.f, 1.f, nm,
                        nm);
#pragma unroll
                for (int u = 0; u < 8; ++u) pv[u] = fast_exp2(tv[u]);
#pragma unroll
                for (int u = 0; u < 8; u += 2) fadd2_acc(rr[u], rr[u + 1], pv[u], pv[u + 1]);
#pragma unroll
                for (int u = 0; u < 8; u += 2) p[(c + u) / 2] = pack_bf16x2(pv[u], pv[u + 1]);
              }
              uint8_t* prow = smem + kPOff + b * kPSlotBytes + a * kPAtomBytes + h * 64;
#pragma unroll
              for (int c = 0; c < 4; ++c)
                *reinterpret_cast<uint4*>(prow + ((c ^ ((h >> 1) & 3)) * 16)) =
                    make_uint4(p[4 * c], p[4 * c + 1], p[4 * c + 2], p[4 * c + 3]);
              // Tokens past the end contribute exactly zero even if the cache
              // tail holds non-finite bytes: clear those V rows of this CTA's
              // stage before its PV reads them (p_full waits for both softmax
              // warps of the step).
              if (a == 1 && nvalid < kStep) {
                uint8_t* vst = smem + kStageOff + (gi % kStages) * kStageBytes;
                const int zrows = kStep - nvalid;  // rows [nvalid, 64) of atoms 0..3
                for (int e = (sub & 1) * 32 + lane; e < zrows * 4 * 8; e += 64) {
                  const int za = e / (zrows * 8), rem = e % (zrows * 8);
                  const int rr2 = nvalid + rem / 8, ch = rem % 8;
                  *reinterpret_cast<uint4*>(vst + za * kKAtomBytes + rr2 * 128 + ch * 16) =
                      make_uint4(0u, 0u, 0u, 0u);
                }
              }
              fence_proxy_async_smem();
              if (a == 1) tc_fence_before();
              __syncwarp();
              if (lane == 0) {
                const int off = b * kPSlotBytes + a * kPAtomBytes + sub * kPWarpBytes;
                bulk_copy_to_peer(peer_p + off, sP + off, kPWarpBytes, peer_xp_full0 + 8u * b);
                if (a == 1) mbar_arrive(bar_p_full(b));
              }
            }
            l += ((rr[0] + rr[1]) + (rr[2] + rr[3])) + ((rr[4] + rr[5]) + (rr[6] + rr[7]));
          }
          if (!ok) break;
          // The row sum over the segment from both parities' shares (each
          // relative to its warp's last reference); the peer gets it for its
          // O rows of these heads.
          {
            float* mine = lpart + ((seg_i & 1) * 2 + par) * kOwn * 2;
            mine[j] = l;
            mine[kOwn + j] = m_known;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_seg_done);
            const bool w = mbar_wait(bar_seg_done, seg_i & 1, abort_flag, err, kSiteXchg, seg_i);
            if (!__all_sync(0xffffffffu, w)) {
              ok = false;
              break;
            }
            const float* s0 = lpart + ((seg_i & 1) * 2) * kOwn * 2;
            const float* s1 = s0 + kOwn * 2;
            const float la = s0[j], ma = s0[kOwn + j], lb = s1[j], mb = s1[kOwn + j];
            const float mf = fmaxf(ma, mb);
            const float lt = (ma == -INFINITY ? 0.f : la * fast_exp2(ma - mf)) +
                             (mb == -INFINITY ? 0.f : lb * fast_exp2(mb - mf));
            if (par == 0)
              st_async_b32(peer_lfin + (seg_i & 1) * kOwn * 4, __float_as_uint(lt),
                           peer_lfin_full0 + 8u * (seg_i & 1));
            prev_m = mf;
            prev_l = lt;
          }
        } else {
          // ================= the peer's heads =================
          // A step of this warp's parity: send this CTA's partial S of these
          // heads to the peer, then take in the peer's P rows of the step: their
          // rescale factors are applied to this CTA's O rows of those heads
          // before the PV of the step may run.
          for (int i = (par - g) & 1; i < n; i += 2) {
            const int gi = g + i;
            const int b = gi & 1;
            bool w = mbar_wait(bar_s_full(b), (gi >> 1) & 1, abort_flag, err, kSiteSFull, gi);
            if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
            tc_fence_after();
            float sv[kStep];
            tmem_ld64(tS + b * 64, sv);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_s_read(b));
            // The peer sends its step gi + 1 into the slot of step gi - 1 only
            // after its softmax has read this CTA's step gi, which is sent
            // only after this CTA's softmax has read the peer's step gi - 1.
            if (gi >= 1) {
              const int gp = gi - 1;
              w = mbar_wait(bar_x_read(gp & 1), (gp >> 1) & 1, abort_flag, err, kSiteXfree, gi);
              if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
            }
#pragma unroll
            for (int hx = 0; hx < 2; ++hx) {
              const uint32_t dst = peer_x + (b * 2 + hx) * kXMsgBytes;
              const uint32_t rbar = peer_x_full0 + 8u * (b * 2 + hx);
#pragma unroll
              for (int c = hx * kXHalf; c < (hx + 1) * kXHalf; c += 4)
                st_async_v4(dst + ((c - hx * kXHalf) / 4) * kXQuadBytes, __float_as_uint(sv[c]),
                            __float_as_uint(sv[c + 1]), __float_as_uint(sv[c + 2]),
                            __float_as_uint(sv[c + 3]), rbar);
            }
            w = mbar_wait<true>(bar_xp_full(b), (gi >> 1) & 1, abort_flag, err, kSitePFull, gi);
            if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
            if (first_of_pair && lane == 0)
              mbar_arrive_expect_tx(bar_xp_full(b), kXpBytes);  // for step gi + 2
            if (i > 0) {
              const float a = alpha_in[b * kOwn + j];
              if (__any_sync(0xffffffffu, a != 1.f)) {
                const int gp = gi - 1;
                w = mbar_wait(bar_kv_empty(gp & (kStages - 1)), (gp / kStages) & 1,
                              abort_flag, err, kSitePvDone, gi);
                if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
                tc_fence_after();
                rescale_o(a);
              }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_p_full(b));
          }
        }
        if (!ok) break;
        prev_b = s.b;
        prev_slot = s.slot;
        prev_seg = seg_i;
        prev_last = g + n - 1;
        g += n;
        ++seg_i;
      }
    }
    if (ok && prev_b >= 0) {
      ok = mbar_wait(bar_kv_empty(prev_last & (kStages - 1)), (prev_last / kStages) & 1,
                     abort_flag, err, kSitePvDone, prev_seg);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        tc_fence_after();
        epilogue();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  // After an abort the peer may have left its loops with a store or copy to
  // this CTA still in flight, one that this CTA never waited for (they land in
  // well under a microsecond).  A CTA that aborted waits 50 us before it
  // arrives at the cluster barrier below, so the peer cannot leave while one
  // of this CTA's own stores or copies is in flight.
  if (*abort_flag) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 50000ull) {
    }
  }
  cluster_sync();  // no CTA leaves while its peer may still touch its smem
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

// ---- combine ------------------------------------------------------------------
// A fixed grid walks the (sequence, head) rows of the sequences the plan
// listed, one warp per row and 16 output columns per lane: empty sequences
// get O = 0, LSE = -inf; cut ones merge their partials,
// L = log sum_s e^{L_s}, O = sum_s e^{L_s - L} O_s.  The plan has already
// found each listed sequence's chunk range, so a row is a few independent
// loads deep.  With nothing listed every block exits at once.
__global__ void __launch_bounds__(256) mla_combine_kernel(
    const int* __restrict__ hdr, const int* __restrict__ bounds, const int4* __restrict__ clist,
    const float* __restrict__ part_lse, const __nv_bfloat16* __restrict__ part_o,
    __nv_bfloat16* __restrict__ o, float* __restrict__ lse) {
  grid_dependency_wait();  // the decode kernel's partials are complete
  const int rows = hdr[4] * kHq;
  const int lane = threadIdx.x & 31;
  const int c0 = lane * 16;
  for (int row = blockIdx.x * 8 + (threadIdx.x >> 5); row < rows; row += gridDim.x * 8) {
    const int4 e = clist[row / kHq];  // {b, k0, k1, first slot}
    const int h = row % kHq;
    const size_t orow = (size_t)e.x * kHq + h;
    uint4* dst = reinterpret_cast<uint4*>(o + orow * kDv + c0);
    if (e.y < 0) {
      dst[0] = make_uint4(0u, 0u, 0u, 0u);
      dst[1] = make_uint4(0u, 0u, 0u, 0u);
      if (lane == 0) lse[orow] = -INFINITY;
      continue;
    }
    const int k0 = e.y, k1 = e.z, s0 = e.w;
    // The chunks over this sequence are merged four at a time: one round of
    // loads for their edges, one for their LSEs and partial rows, then a
    // running-max merge (O = sum w_k O_k / sum w_k, w_k = e^(lse_k - max)).
    // Empty chunks wrote nothing and chunks with LSE = -inf weigh nothing.
    float mx = -INFINITY, wsum = 0.f;
    float acc[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) acc[c] = 0.f;
    for (int kb = k0; kb <= k1; kb += 4) {
      int nz[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int k = kb + u;
        nz[u] = (k <= k1) ? bounds[k + 1] - bounds[k] : 0;
      }
      float ls[4];
      uint4 v[4][2];  // 16 bf16 partial values a lane
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int k = kb + u;
        const int slot = (k == k0) ? s0 : 2 * k;
        ls[u] = -INFINITY;
        if (nz[u] > 0) {
          ls[u] = part_lse[(size_t)slot * kHq + h];
          const uint4* src =
              reinterpret_cast<const uint4*>(part_o + ((size_t)slot * kHq + h) * kDv + c0);
          v[u][0] = src[0];
          v[u][1] = src[1];
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (ls[u] == -INFINITY) continue;
        const float m_new = fmaxf(mx, ls[u]);
        const float a = expf(mx - m_new);  // 0 while mx is still -inf
        const float w = expf(ls[u] - m_new);
        wsum = wsum * a + w;
        const uint32_t* pw = reinterpret_cast<const uint32_t*>(v[u]);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float2 f = unpack_bf16x2(pw[q]);
          acc[2 * q] = acc[2 * q] * a + w * f.x;
          acc[2 * q + 1] = acc[2 * q + 1] * a + w * f.y;
        }
        mx = m_new;
      }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
    for (int q = 0; q < 2; ++q)
      dst[q] = make_uint4(pack_bf16x2(acc[8 * q] * inv, acc[8 * q + 1] * inv),
                          pack_bf16x2(acc[8 * q + 2] * inv, acc[8 * q + 3] * inv),
                          pack_bf16x2(acc[8 * q + 4] * inv, acc[8 * q + 5] * inv),
                          pack_bf16x2(acc[8 * q + 6] * inv, acc[8 * q + 7] * inv));
    if (lane == 0) lse[orow] = (wsum > 0.f) ? mx + logf(wsum) : -INFINITY;
  }
}

// The latent pool as a 2-D tensor [rows, 576]: boxes of `box_cols` columns x
// `box_rows` rows with 128-byte (64 columns) or 64-byte (32 columns) swizzle.
CUresult make_map_2d(CUtensorMap* map, const void* ptr, long long rows, int box_rows,
                     int box_cols) {
  PFN_encodeTiled enc = get_encode_tiled();
  if (!enc) return CUDA_ERROR_NOT_FOUND;
  cuuint64_t dims[2] = {(cuuint64_t)kDk, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kDk * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle sw =
      box_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// Clusters of two that can be resident at once (cached per device).
int active_clusters(int num_sms) {
  static int cached[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return num_sms / 2;
  std::lock_guard<std::mutex> lk(mu);
  if (cached[dev] == 0) {
    int n = 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, mla_decode_kernel, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = num_sms / 2;
    }
    cached[dev] = n < num_sms / 2 ? n : num_sms / 2;
  }
  return cached[dev];
}

}  // namespace

size_t mla_workspace_bytes(int B, int Hq, int max_blocks, int num_sms, int pages_per_split) {
  (void)Hq;
  return ws_layout(B, max_chunks_for(B, max_blocks, num_sms, pages_per_split)).total;
}

cudaError_t launch_mla_decode(const MlaArgs& a, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(mla_decode_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const int clusters = active_clusters(a.num_sms);
  const WsLayout w = ws_layout(a.B, max_chunks_for(a.B, a.max_blocks, a.num_sms, a.pages_per_split));
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  int* hdr = reinterpret_cast<int*>(ws + w.header);
  int* prefix = reinterpret_cast<int*>(ws + w.prefix);
  int* bounds = reinterpret_cast<int*>(ws + w.bounds);
  int* cstart = reinterpret_cast<int*>(ws + w.cstart);
  int4* clist = reinterpret_cast<int4*>(ws + w.clist);
  float* plse = reinterpret_cast<float*>(ws + w.plse);
  __nv_bfloat16* po = reinterpret_cast<__nv_bfloat16*>(ws + w.po);

  CUtensorMap mkv, mrope;
  CUresult r = make_map_2d(&mkv, a.kv, (long long)a.num_blocks * kPage, kStep, 64);
  if (r == CUDA_SUCCESS)
    r = make_map_2d(&mrope, a.kv, (long long)a.num_blocks * kPage, kStep, kRopeCols);
  if (r != CUDA_SUCCESS) {
    attn_set_error("mla_decode: cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return cudaErrorInvalidValue;
  }
  {
    cudaLaunchAttribute pdl1[1];
    pdl1[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl1[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t pc = {};
    pc.gridDim = dim3(1, 1, 1);
    pc.blockDim = dim3(1024, 1, 1);
    pc.stream = s;
    pc.attrs = pdl1;
    pc.numAttrs = 1;
    e = cudaLaunchKernelEx(&pc, mla_plan_kernel, (const int32_t*)a.seqlens, a.B, a.max_blocks,
                           clusters, a.pages_per_split, hdr, prefix, bounds, cstart, clist,
                           a.err);
    if (e != cudaSuccess) return e;
  }
  const float scale_log2 = a.scale * 1.4426950408889634f;
  // decode and combine are launched as programmatic dependents of the kernel
  // before them: each starts while its predecessor finishes and waits for it
  // (griddepcontrol.wait) only where it reads that kernel's output
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, mla_decode_kernel, mkv, mrope,
                         static_cast<const __nv_bfloat16*>(a.q), a.block_table, a.seqlens,
                         static_cast<__nv_bfloat16*>(a.o), a.lse, (const int*)hdr,
                         (const int*)prefix, (const int*)bounds, (const int*)cstart, plse, po,
                         a.B, a.max_blocks,
                         a.num_blocks, scale_log2, a.err, a.debug_skip_step);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(4 * a.num_sms, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = 0;
  e = cudaLaunchKernelEx(&cfg, mla_combine_kernel, (const int*)hdr, (const int*)bounds,
                         (const int4*)clist, (const float*)plse, (const __nv_bfloat16*)po,
                         static_cast<__nv_bfloat16*>(a.o), a.lse);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// ---- fixed scratch for callers that cannot allocate ---------------------------
// mla_decode_noalloc runs the same plan / decode / combine kernels with the
// workspace placed in this file-scope device array instead of a caller
// buffer.  Its size covers the automatic plan for up to kNoAllocMaxBatch
// sequences on a device of up to kNoAllocMaxSms SMs (at most one chunk per
// 2-SM cluster, two partial slots per chunk).  Every GPU that loads the
// library reserves it until exit.
namespace {
constexpr int kNoAllocMaxBatch = 8192;
constexpr int kNoAllocMaxSms = 160;
constexpr size_t kNoAllocScratchBytes = ws_layout(kNoAllocMaxBatch, kNoAllocMaxSms / 2).total;
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
