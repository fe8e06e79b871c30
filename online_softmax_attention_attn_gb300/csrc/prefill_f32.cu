// prefill_f32.cu -- fp32 attention forward on CUDA cores (FFMA), sm_103a.
//
// Loop order and state follow the "FP32 CUDA-core FlashAttention-2 v2" blog
// (dandandamowang post_1787450400): one CTA owns a block of Br query rows
// (section 1.1), Q stays in shared memory for the whole KV loop and m/l/O stay
// on chip (section 1.2), O is rescaled with exp(m_old - m_new) and divided by
// l once at the end (section 1.3), KV blocks above the diagonal are never
// visited and only blocks crossing it are masked element by element
// (sections 1.4 and 3.4), K/V blocks are prefetched with cp.async and
// zero-filled past N while those keys get -inf (section 3.2).
//
// What differs from the blog's kernel: instead of one thread per query row
// (latency bound, section 4.2), 256 threads form a 16 x 16 grid and each
// thread owns an 8-row x 4-key tile of S and an 8-row x 4-column tile of O,
// so every shared-memory load feeds 8-32 FMAs.  Rows are interleaved
// (r = ty + 16 i) and keys too (c = tx + 16 j), which makes the padded
// 68-float rows bank-conflict free for 128-bit loads.  Both products use the
// packed two-lane FMA (fma.rn.f32x2), half the instructions of scalar FFMAs:
// S over pairs of d (even and odd partial sums per element, added at the
// end), PV over pairs of output columns, each P value (stored once in shared
// memory) multiplying both lanes.  Shared-memory loads, not the FMA pipe, set
// the pace of these loops, so P is not stored twice as a (p, p) pair and
// both loops are unrolled eight steps deep.  Softmax runs in base 2 with
// log2(e) folded into the Q pre-scale.  The CTA's two halves (warps 0-3 and
// 4-7, 64 interleaved rows each) synchronise only among themselves and run
// the KV loop half a block apart, so that one half's softmax overlaps the
// other half's FMA loops: K/V blocks sit in a ring of four buffers whose
// loads report on a full mbarrier (cp.async.mbarrier.arrive) and whose reuse
// waits on an empty one.  Each block is loaded one block ahead; the fourth
// buffer is slack that lets the leading half run up to three blocks ahead of
// the other (against three buffers: 2-3 % faster).  Every wait is bounded; a
// stuck pipeline records ATTN_ERR_DEVICE_TIMEOUT.
// Blocks are 128 query rows; a grid of fewer (head, block) pairs than half
// the SMs runs with 32-row blocks instead (same 256 threads, two rows each),
// so that a small problem spreads over four times as many SMs.
#include <math.h>

#include "common.cuh"

namespace {

constexpr int kD = 64;
constexpr int kBrLarge = 128;          // query rows per CTA (a 32-row variant serves small grids)
constexpr int kBrSmall = 32;
constexpr int kBc = 64;
constexpr int kThreads = 256;
constexpr int kTy = 16;                 // row groups (rows interleaved by kTy)
constexpr int kKvBufs = 4;              // K/V blocks in shared memory
constexpr int kQPad = kD + 4;  // 68 floats: 16-byte aligned rows, shifted banks
constexpr int kKPad = kD + 4;
constexpr int kPPad = kBc + 16;  // P: 80 floats a row (the two rows of a warp 16 banks apart)
template <int kBr>
constexpr int smem_bytes() {
  return (kBr * kQPad + kKvBufs * kBc * kKPad + kKvBufs * kBc * kD + kBr * kPPad) * 4 +
         (2 * kKvBufs + 1) * 8 + 16;  // + barriers, abort flag
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}
// Arrive on `bar` once every cp.async this thread has issued so far has
// landed (the arrival is one of the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Copy one K and one V block [kv0, kv0 + Bc) of head bh into buffer `buf`.
// Rows at or past N are zero-filled (their scores are masked to -inf).
__device__ __forceinline__ void load_kv_block(const float* __restrict__ kg,
                                              const float* __restrict__ vg, float* Ks,
                                              float* Vs, int kv0, int N, int buf) {
  constexpr int kVecPerRow = kD / 4;
  constexpr int kVecs = kBc * kVecPerRow;  // 1024 16-byte chunks per tensor
#pragma unroll
  for (int it = 0; it < kVecs / kThreads; ++it) {
    int i = threadIdx.x + it * kThreads;
    int row = i / kVecPerRow, c4 = i % kVecPerRow;
    int key = kv0 + row;
    bool ok = key < N;
    int src_row = ok ? key : (N - 1);
    uint32_t kd = gb300::smem_u32(Ks + (buf * kBc + row) * kKPad + c4 * 4);
    uint32_t vd = gb300::smem_u32(Vs + (buf * kBc + row) * kD + c4 * 4);
    cp_async16(kd, kg + (size_t)src_row * kD + c4 * 4, ok);
    cp_async16(vd, vg + (size_t)src_row * kD + c4 * 4, ok);
  }
}

template <int kBr, bool kCausal>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                       const float* __restrict__ v, float* __restrict__ o,
                       float* __restrict__ lse, int BH, int N, float qscale, int* err,
                       int debug_skip_block) {
  constexpr int kRows = kBr / kTy;  // query rows per thread
  extern __shared__ __align__(16) float smem[];
  float* Qs = smem;                       // [Br][68], pre-scaled by scale*log2(e)
  float* Ks = Qs + kBr * kQPad;           // [4][Bc][68]
  float* Vs = Ks + kKvBufs * kBc * kKPad; // [4][Bc][64]
  float* Ps = Vs + kKvBufs * kBc * kD;    // [Br][80]: P of the current block
  uint64_t* bars = reinterpret_cast<uint64_t*>(Ps + kBr * kPPad);  // full[4], empty[4], go
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kKvBufs + 1);
  const uint32_t bar0 = gb300::smem_u32(bars);
  auto bar_full = [&](int b) { return bar0 + 8u * b; };
  auto bar_empty = [&](int b) { return bar0 + 8u * (kKvBufs + b); };
  const uint32_t bar_go = bar0 + 8u * (2 * kKvBufs);

  const int n_qt = (N + kBr - 1) / kBr;
  // Heaviest causal Q blocks first across all heads (longest-first order).
  const int lin = blockIdx.x;
  const int qt = kCausal ? (n_qt - 1 - lin / BH) : (lin / BH);
  const int bh = lin % BH;
  const int q0 = qt * kBr;

  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  // The two halves of the CTA (warps 0-3: ty 0-7, warps 4-7: ty 8-15) own
  // disjoint rows and run the block loop half a block apart, so that one
  // half's softmax overlaps the other's FMA loops.
  const int half = ty >> 3;

  if (tid == 0) {
    for (int b = 0; b < kKvBufs; ++b) {
      gb300::mbar_init(bar_full(b), kThreads);   // every thread's copies of the block
      gb300::mbar_init(bar_empty(b), kThreads);  // every thread done reading it
    }
    gb300::mbar_init(bar_go, kThreads / 2);      // half 0 has finished its first softmax
    *abort_flag = 0;
    gb300::fence_mbar_init();
  }

  const size_t head = (size_t)bh * N * kD;
  const float* qg = q + head;
  const float* kg = k + head;
  const float* vg = v + head;

  // Q block -> shared (once), scaled so that S comes out in log2 units.
  for (int i = tid; i < kBr * (kD / 4); i += kThreads) {
    int row = i / (kD / 4), c4 = i % (kD / 4);
    float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
    if (q0 + row < N) {
      val = *reinterpret_cast<const float4*>(qg + (size_t)(q0 + row) * kD + c4 * 4);
      val.x *= qscale; val.y *= qscale; val.z *= qscale; val.w *= qscale;
    }
    *reinterpret_cast<float4*>(Qs + row * kQPad + c4 * 4) = val;
  }
  __syncthreads();  // Q and the barriers are ready

  const int kv_limit = kCausal ? min(q0 + kBr, N) : N;
  const int Tc = (kv_limit + kBc - 1) / kBc;

  float m_i[kRows], l_i[kRows], acc[kRows][4];
#pragma unroll
  for (int i = 0; i < kRows; ++i) {
    m_i[i] = -INFINITY;
    l_i[i] = 0.f;
#pragma unroll
    for (int d = 0; d < 4; ++d) acc[i][d] = 0.f;
  }

  // Each thread copies its share of every K/V block and reports completion
  // on the block's full barrier; block j lives in buffer j % 4.
  auto issue_load = [&](int jb) {
    if (jb == debug_skip_block) return;  // test hook: this block never arrives
    load_kv_block(kg, vg, Ks, Vs, jb * kBc, N, jb % kKvBufs);
    cp_async_arrive(bar_full(jb % kKvBufs));
  };
  issue_load(0);
  bool ok = true;
  if (half == 1)
    ok = gb300::mbar_wait(bar_go, 0, abort_flag, err, gb300::kSiteQFull, 0);

  for (int j = 0; j < Tc; ++j) {
    const int buf = j % kKvBufs;
    const int kv0 = j * kBc;
    if (ok && j + 1 < Tc) {
      // block j+1 goes where block j-3 was: every thread must be done with it
      const int nb = (j + 1) % kKvBufs;
      if (j + 1 >= kKvBufs)
        ok = gb300::mbar_wait(bar_empty(nb), ((j + 1) / kKvBufs - 1) & 1, abort_flag, err,
                              gb300::kSiteKvEmpty, j);
      if (ok) issue_load(j + 1);
    }
    if (ok) ok = gb300::mbar_wait(bar_full(buf), (j / kKvBufs) & 1, abort_flag, err,
                                  gb300::kSiteKvFull, j);
    // One barrier of the half per block, after its waits (all bounded): the
    // half leaves the loop together if any wait of the CTA has failed, and
    // every thread of the half is done reading P of block j-1 (its PV).
    if (gb300::named_barrier_any(1 + half, kThreads / 2, !ok || *abort_flag != 0)) {
      ok = false;
      break;
    }

    // ---- S = Q K^T for this thread's 8 x 4 tile (log2 units).  Packed
    // two-lane FMAs over pairs of d: each (row, key) keeps an even-d and an
    // odd-d partial sum, added once at the end.
    float se[kRows][4], so[kRows][4];
#pragma unroll
    for (int i = 0; i < kRows; ++i)
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) se[i][jj] = so[i][jj] = 0.f;
    const float* Kb = Ks + buf * kBc * kKPad;
#pragma unroll 8
    for (int d4 = 0; d4 < kD / 4; ++d4) {
      float4 qv[kRows], kv4[4];
#pragma unroll
      for (int i = 0; i < kRows; ++i)
        qv[i] = *reinterpret_cast<const float4*>(Qs + (ty + kTy * i) * kQPad + d4 * 4);
#pragma unroll
      for (int jj = 0; jj < 4; ++jj)
        kv4[jj] = *reinterpret_cast<const float4*>(Kb + (tx + 16 * jj) * kKPad + d4 * 4);
#pragma unroll
      for (int i = 0; i < kRows; ++i)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          gb300::ffma2(se[i][jj], so[i][jj], qv[i].x, qv[i].y, kv4[jj].x, kv4[jj].y, se[i][jj],
                       so[i][jj]);
          gb300::ffma2(se[i][jj], so[i][jj], qv[i].z, qv[i].w, kv4[jj].z, kv4[jj].w, se[i][jj],
                       so[i][jj]);
        }
    }
    float s[kRows][4];
#pragma unroll
    for (int i = 0; i < kRows; ++i)
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) s[i][jj] = se[i][jj] + so[i][jj];

    // ---- mask: keys past N; causal diagonal block: key > row
    const bool tail = kv0 + kBc > N;
    const bool diag = kCausal && (kv0 + kBc - 1 > q0);
    if (tail || diag) {
#pragma unroll
      for (int i = 0; i < kRows; ++i)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          int key = kv0 + tx + 16 * jj;
          int row = q0 + ty + kTy * i;
          if (key >= N || (kCausal && key > row)) s[i][jj] = -INFINITY;
        }
    }

    // ---- online softmax (base 2): m, rescale factors, P, l
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
      float mt = fmaxf(fmaxf(s[i][0], s[i][1]), fmaxf(s[i][2], s[i][3]));
#pragma unroll
      for (int off = 8; off > 0; off >>= 1)
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
      const float m_new = fmaxf(m_i[i], mt);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = gb300::fast_exp2(m_i[i] - m_use);
      float rs = 0.f;
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        s[i][jj] = gb300::fast_exp2(s[i][jj] - m_use);
        rs += s[i][jj];
      }
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) rs += __shfl_xor_sync(0xffffffffu, rs, off);
      l_i[i] = alpha * l_i[i] + rs;
      m_i[i] = m_new;
#pragma unroll
      for (int d = 0; d < 4; ++d) acc[i][d] *= alpha;
#pragma unroll
      for (int jj = 0; jj < 4; ++jj)
        Ps[(ty + kTy * i) * kPPad + tx + 16 * jj] = s[i][jj];
    }
    gb300::named_barrier_sync(1 + half, kThreads / 2);  // the half's P rows are visible
    if (j == 0 && half == 0) gb300::mbar_arrive(bar_go);

    // ---- O += P V for this thread's 8 x 4 tile: packed two-lane FMAs over
    // pairs of output columns, one P value for both lanes
    const float* Vb = Vs + buf * kBc * kD;
#pragma unroll 8
    for (int c4 = 0; c4 < kBc / 4; ++c4) {
      float4 pa[kRows], vv[4];
#pragma unroll
      for (int i = 0; i < kRows; ++i)
        pa[i] = *reinterpret_cast<const float4*>(Ps + (ty + kTy * i) * kPPad + c4 * 4);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        vv[kk] = *reinterpret_cast<const float4*>(Vb + (c4 * 4 + kk) * kD + tx * 4);
#pragma unroll
      for (int i = 0; i < kRows; ++i) {
        gb300::ffma2(acc[i][0], acc[i][1], pa[i].x, pa[i].x, vv[0].x, vv[0].y, acc[i][0], acc[i][1]);
        gb300::ffma2(acc[i][2], acc[i][3], pa[i].x, pa[i].x, vv[0].z, vv[0].w, acc[i][2], acc[i][3]);
        gb300::ffma2(acc[i][0], acc[i][1], pa[i].y, pa[i].y, vv[1].x, vv[1].y, acc[i][0], acc[i][1]);
        gb300::ffma2(acc[i][2], acc[i][3], pa[i].y, pa[i].y, vv[1].z, vv[1].w, acc[i][2], acc[i][3]);
        gb300::ffma2(acc[i][0], acc[i][1], pa[i].z, pa[i].z, vv[2].x, vv[2].y, acc[i][0], acc[i][1]);
        gb300::ffma2(acc[i][2], acc[i][3], pa[i].z, pa[i].z, vv[2].z, vv[2].w, acc[i][2], acc[i][3]);
        gb300::ffma2(acc[i][0], acc[i][1], pa[i].w, pa[i].w, vv[3].x, vv[3].y, acc[i][0], acc[i][1]);
        gb300::ffma2(acc[i][2], acc[i][3], pa[i].w, pa[i].w, vv[3].z, vv[3].w, acc[i][2], acc[i][3]);
      }
    }
    gb300::mbar_arrive(bar_empty(buf));  // this thread is done with block j's K and V
  }
  // Half 0 may have stopped before letting half 1 start.
  if (half == 0 && Tc == 0) gb300::mbar_arrive(bar_go);
  cp_async_wait_all();  // every copy this thread started has landed

  // ---- epilogue: O = O / l (one division per row), LSE, single HBM write
  if (!ok) return;
  constexpr float kLn2 = 0.69314718055994530942f;
#pragma unroll
  for (int i = 0; i < kRows; ++i) {
    const int row = q0 + ty + kTy * i;
    if (row >= N) continue;
    const float inv_l = 1.0f / l_i[i];
    float4 out = make_float4(acc[i][0] * inv_l, acc[i][1] * inv_l, acc[i][2] * inv_l,
                             acc[i][3] * inv_l);
    *reinterpret_cast<float4*>(o + head + (size_t)row * kD + tx * 4) = out;
    if (tx == 0) lse[(size_t)bh * N + row] = (m_i[i] + log2f(l_i[i])) * kLn2;
  }
}

}  // namespace

bool prefill_f32_info(int D, int* Br, int* Bc, int* threads, int* smem) {
  if (D != kD) return false;
  if (Br) *Br = kBrLarge;
  if (Bc) *Bc = kBc;
  if (threads) *threads = kThreads;
  if (smem) *smem = smem_bytes<kBrLarge>();
  return true;
}

namespace {

int sm_count() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    cached[dev] = n;
  }
  return cached[dev];
}

template <int kBr>
cudaError_t launch_br(const PrefillF32Args& a, cudaStream_t s) {
  const int BH = a.B * a.H;
  const int n_qt = (a.N + kBr - 1) / kBr;
  const long long blocks = (long long)n_qt * BH;
  if (blocks > 0x7fffffffLL) {
    attn_set_error("attn_fwd: too many query blocks (%lld)", blocks);
    return cudaErrorInvalidValue;
  }
  const float qscale = a.scale * 1.4426950408889634f;  // log2(e)
  constexpr int kSmem = smem_bytes<kBr>();
  auto kern = a.causal ? prefill_f32_kernel<kBr, true> : prefill_f32_kernel<kBr, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)blocks, kThreads, kSmem, s>>>(a.q, a.k, a.v, a.o, a.lse, BH, a.N, qscale,
                                                  a.err, a.debug_skip_block);
  return cudaGetLastError();
}

}  // namespace

// 128-row blocks, unless they would leave most of the GPU idle (fewer CTAs
// than half its SMs): then 32-row blocks, four times as many CTAs each with
// a quarter of the work per KV block.
cudaError_t launch_prefill_f32(const PrefillF32Args& a, cudaStream_t s) {
  const long long large = (long long)((a.N + kBrLarge - 1) / kBrLarge) * a.B * a.H;
  const int nsm = sm_count();
  if (nsm > 0 && 2 * large < nsm) return launch_br<kBrSmall>(a, s);
  return launch_br<kBrLarge>(a, s);
}
