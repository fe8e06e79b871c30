// prefill_f32.cu -- fp32 attention forward on CUDA cores (FFMA), sm_103a.
//
// Loop order and state follow the "FP32 CUDA-core FlashAttention-2 v2" blog
// (dandandamowang post_1787450400): one CTA owns a block of Br query rows
// (section 1.1), Q stays in shared memory for the whole KV loop and m/l/O stay
// on chip (section 1.2), O is rescaled with exp(m_old - m_new) and divided by
// l once at the end (section 1.3), KV blocks above the diagonal are never
// visited and only blocks crossing it are masked element by element
// (sections 1.4 and 3.4), K/V blocks are double buffered with cp.async and
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
// end), PV over pairs of output columns with P kept in shared memory as
// (p, p) pairs.  Softmax runs in base 2 with log2(e) folded into the Q
// pre-scale.
#include <math.h>

#include "common.cuh"

namespace {

constexpr int kD = 64;
constexpr int kBr = 128;
constexpr int kBc = 64;
constexpr int kThreads = 256;
constexpr int kQPad = kD + 4;  // 68 floats: 16-byte aligned rows, shifted banks
constexpr int kKPad = kD + 4;
constexpr int kPPad = 2 * kBc + 8;  // P stored as (p, p) pairs: 136 floats a row
constexpr int kSmemFloats = kBr * kQPad + 2 * kBc * kKPad + 2 * kBc * kD + kBr * kPPad;
constexpr int kSmemBytes = kSmemFloats * 4;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
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

template <bool kCausal>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                       const float* __restrict__ v, float* __restrict__ o,
                       float* __restrict__ lse, int BH, int N, float qscale) {
  extern __shared__ __align__(16) float smem[];
  float* Qs = smem;                       // [Br][68], pre-scaled by scale*log2(e)
  float* Ks = Qs + kBr * kQPad;           // [2][Bc][68]
  float* Vs = Ks + 2 * kBc * kKPad;       // [2][Bc][64]
  float* Ps = Vs + 2 * kBc * kD;          // [Br][136]: each P twice, (p, p)

  const int n_qt = (N + kBr - 1) / kBr;
  // Heaviest causal Q blocks first across all heads (longest-first order).
  const int lin = blockIdx.x;
  const int qt = kCausal ? (n_qt - 1 - lin / BH) : (lin / BH);
  const int bh = lin % BH;
  const int q0 = qt * kBr;

  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;

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

  const int kv_limit = kCausal ? min(q0 + kBr, N) : N;
  const int Tc = (kv_limit + kBc - 1) / kBc;

  float m_i[8], l_i[8], acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    m_i[i] = -INFINITY;
    l_i[i] = 0.f;
#pragma unroll
    for (int d = 0; d < 4; ++d) acc[i][d] = 0.f;
  }

  load_kv_block(kg, vg, Ks, Vs, 0, N, 0);
  cp_async_commit();

  for (int j = 0; j < Tc; ++j) {
    const int buf = j & 1;
    const int kv0 = j * kBc;
    cp_async_wait_all();
    __syncthreads();  // block j visible; everyone is done with block j-1
    if (j + 1 < Tc) {
      load_kv_block(kg, vg, Ks, Vs, kv0 + kBc, N, buf ^ 1);
      cp_async_commit();
    }

    // ---- S = Q K^T for this thread's 8 x 4 tile (log2 units).  Packed
    // two-lane FMAs over pairs of d: each (row, key) keeps an even-d and an
    // odd-d partial sum, added once at the end.
    float se[8][4], so[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) se[i][jj] = so[i][jj] = 0.f;
    const float* Kb = Ks + buf * kBc * kKPad;
#pragma unroll 4
    for (int d4 = 0; d4 < kD / 4; ++d4) {
      float4 qv[8], kv4[4];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        qv[i] = *reinterpret_cast<const float4*>(Qs + (ty + 16 * i) * kQPad + d4 * 4);
#pragma unroll
      for (int jj = 0; jj < 4; ++jj)
        kv4[jj] = *reinterpret_cast<const float4*>(Kb + (tx + 16 * jj) * kKPad + d4 * 4);
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          gb300::ffma2(se[i][jj], so[i][jj], qv[i].x, qv[i].y, kv4[jj].x, kv4[jj].y, se[i][jj],
                       so[i][jj]);
          gb300::ffma2(se[i][jj], so[i][jj], qv[i].z, qv[i].w, kv4[jj].z, kv4[jj].w, se[i][jj],
                       so[i][jj]);
        }
    }
    float s[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) s[i][jj] = se[i][jj] + so[i][jj];

    // ---- mask: keys past N; causal diagonal block: key > row
    const bool tail = kv0 + kBc > N;
    const bool diag = kCausal && (kv0 + kBc - 1 > q0);
    if (tail || diag) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          int key = kv0 + tx + 16 * jj;
          int row = q0 + ty + 16 * i;
          if (key >= N || (kCausal && key > row)) s[i][jj] = -INFINITY;
        }
    }

    // ---- online softmax (base 2): m, rescale factors, P, l
#pragma unroll
    for (int i = 0; i < 8; ++i) {
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
        *reinterpret_cast<float2*>(Ps + (ty + 16 * i) * kPPad + 2 * (tx + 16 * jj)) =
            make_float2(s[i][jj], s[i][jj]);
    }
    __syncthreads();  // P visible

    // ---- O += P V for this thread's 8 x 4 tile: packed two-lane FMAs over
    // pairs of output columns, P read as (p, p) pairs
    const float* Vb = Vs + buf * kBc * kD;
#pragma unroll 2
    for (int c4 = 0; c4 < kBc / 4; ++c4) {
      float4 pa[8], pb[8], vv[4];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        pa[i] = *reinterpret_cast<const float4*>(Ps + (ty + 16 * i) * kPPad + c4 * 8);
        pb[i] = *reinterpret_cast<const float4*>(Ps + (ty + 16 * i) * kPPad + c4 * 8 + 4);
      }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        vv[kk] = *reinterpret_cast<const float4*>(Vb + (c4 * 4 + kk) * kD + tx * 4);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        gb300::ffma2(acc[i][0], acc[i][1], pa[i].x, pa[i].y, vv[0].x, vv[0].y, acc[i][0], acc[i][1]);
        gb300::ffma2(acc[i][2], acc[i][3], pa[i].x, pa[i].y, vv[0].z, vv[0].w, acc[i][2], acc[i][3]);
        gb300::ffma2(acc[i][0], acc[i][1], pa[i].z, pa[i].w, vv[1].x, vv[1].y, acc[i][0], acc[i][1]);
        gb300::ffma2(acc[i][2], acc[i][3], pa[i].z, pa[i].w, vv[1].z, vv[1].w, acc[i][2], acc[i][3]);
        gb300::ffma2(acc[i][0], acc[i][1], pb[i].x, pb[i].y, vv[2].x, vv[2].y, acc[i][0], acc[i][1]);
        gb300::ffma2(acc[i][2], acc[i][3], pb[i].x, pb[i].y, vv[2].z, vv[2].w, acc[i][2], acc[i][3]);
        gb300::ffma2(acc[i][0], acc[i][1], pb[i].z, pb[i].w, vv[3].x, vv[3].y, acc[i][0], acc[i][1]);
        gb300::ffma2(acc[i][2], acc[i][3], pb[i].z, pb[i].w, vv[3].z, vv[3].w, acc[i][2], acc[i][3]);
      }
    }
  }

  // ---- epilogue: O = O / l (one division per row), LSE, single HBM write
  constexpr float kLn2 = 0.69314718055994530942f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int row = q0 + ty + 16 * i;
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
  if (Br) *Br = kBr;
  if (Bc) *Bc = kBc;
  if (threads) *threads = kThreads;
  if (smem) *smem = kSmemBytes;
  return true;
}

cudaError_t launch_prefill_f32(const PrefillF32Args& a, cudaStream_t s) {
  const int BH = a.B * a.H;
  const int n_qt = (a.N + kBr - 1) / kBr;
  const long long blocks = (long long)n_qt * BH;
  if (blocks > 0x7fffffffLL) {
    attn_set_error("attn_fwd: too many query blocks (%lld)", blocks);
    return cudaErrorInvalidValue;
  }
  const float qscale = a.scale * 1.4426950408889634f;  // log2(e)
  cudaError_t e;
  if (a.causal) {
    e = cudaFuncSetAttribute(prefill_f32_kernel<true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    prefill_f32_kernel<true><<<(unsigned)blocks, kThreads, kSmemBytes, s>>>(
        a.q, a.k, a.v, a.o, a.lse, BH, a.N, qscale);
  } else {
    e = cudaFuncSetAttribute(prefill_f32_kernel<false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    prefill_f32_kernel<false><<<(unsigned)blocks, kThreads, kSmemBytes, s>>>(
        a.q, a.k, a.v, a.o, a.lse, BH, a.N, qscale);
  }
  return cudaGetLastError();
}
