// mla_absorb.cu -- the two projections around MLA absorbed decode.
//
// The "MLA x FlashAttention-3 fusion" article (hnwysp news 119127) folds the
// per-head up-projections into the query and the output: with the latent
// row c_t (512) and per-head W_UK, W_UV, the score of head h is
//   q_nope_h . (W_UK_h^T c_t) + q_rope_h . k_rope_t = (q_nope_h W_UK_h) . c_t + ...
// (the absorption identity), and its output is (sum_t p_t c_t) W_UV_h.  So
// the decode kernel needs the absorbed query [q_nope_h W_UK_h | q_rope_h]
// (576 wide) and leaves a 512-wide latent output that W_UV_h maps to the
// head's values.  Both are per-head products Y_h = X_h W_h of a few token
// rows X_h with a per-head weight matrix W_h.
//
// GB300 design: one CTA per (head, 128 output columns, 64 tokens) computes
// Y_h^T = W_h^T X_h^T on the tensor cores (tcgen05.mma kind::f16, M = 128
// output columns, N = 64 tokens, fp32 accumulators in TMEM).  W_h is read in
// its row-major [k][m] layout as an MN-major A operand and X_h as a K-major B
// operand, both TMA-loaded with the 128-byte swizzle in 64-wide chunks of k,
// each chunk on its own mbarrier so the MMAs start as soon as the first one
// lands.  Every weight byte is read once (the work is bound by the weights'
// HBM traffic); tokens past B are zero-filled by TMA and never stored.  The
// absorbing call also copies q_rope into the last entries of each row.
#include <math.h>

#include "common.cuh"

namespace {

using namespace gb300;

constexpr int kThreads = 128;        // 4 warps: TMEM lanes = output columns
constexpr int kTileM = 128;          // output columns per CTA
constexpr int kTileN = 64;           // tokens per CTA
constexpr int kMaxK = 512;           // reduction width (q_nope 128, latent 512)
constexpr int kChunk = 64;           // k per TMA chunk (one 128-byte row)
constexpr int kChunkBytes = kChunk * 128;  // a [64 rows][128 B] swizzled block

// shared memory: W as 2 atoms of 64 output columns, each [K rows][128 B];
// X as K/64 chunks of [64 tokens][128 B]; then the barriers.
constexpr int smem_bytes(int K) {
  return 2 * K * 128 + (K / kChunk) * kChunkBytes + (K / kChunk + 1) * 8 + 16 + 1024;
}

__global__ void __launch_bounds__(kThreads, 1)
    mla_proj_kernel(const __grid_constant__ CUtensorMap tmW,
                    const __grid_constant__ CUtensorMap tmX, __nv_bfloat16* __restrict__ y,
                    int ldy, const __nv_bfloat16* __restrict__ rope, int d_rope, int rope_off,
                    int B, int Hq, int K, int M, int* err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const int nchunks = K / kChunk;
  const uint32_t sW = base;                   // atom a at + a * K * 128
  const uint32_t sX = base + 2 * K * 128;     // chunk c at + c * kChunkBytes
  const uint32_t bars = sX + nchunks * kChunkBytes;
  auto bar_full = [&](int c) { return bars + 8u * c; };
  const uint32_t bar_done = bars + 8u * nchunks;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + (bars - base) + 8 * (nchunks + 1));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int h = blockIdx.x, m0 = blockIdx.y * kTileM, b0 = blockIdx.z * kTileN;
  const int warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    for (int c = 0; c <= nchunks; ++c) mbar_init(bars + 8u * c, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmW);
    prefetch_tmap(&tmX);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), kTileN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tD = *tmem_slot;
  // launched as a programmatic dependent: the set-up above overlaps the
  // previous kernel on the stream, whose writes are read only from here on
  grid_dependency_wait();
  grid_launch_dependents();

  if (threadIdx.x == 0) {
    // every chunk's loads at once, each chunk on its own barrier
    for (int c = 0; c < nchunks; ++c) {
      mbar_arrive_expect_tx(bar_full(c), 3 * kChunkBytes);
      for (int a = 0; a < 2; ++a)
        tma_load_3d(sW + a * K * 128 + c * kChunkBytes, &tmW, bar_full(c), m0 + a * 64,
                    c * kChunk, h);
      tma_load_3d(sX + c * kChunkBytes, &tmX, bar_full(c), c * kChunk, h, b0);
    }
    // D[m][b] += W[k][m] X[b][k]: A = W (MN-major: the two 64-column atoms
    // K * 128 bytes apart, 8-row groups 1024 apart), B = X (K-major)
    constexpr uint32_t kIdesc = idesc_bf16(kTileM, kTileN, true, false);
    const uint64_t ad0 = sdesc_sw128(sW, K * 128, 1024);
    const uint64_t bd0 = sdesc_sw128(sX, 16, 1024);
    bool ok = true;
    for (int c = 0; c < nchunks && ok; ++c) {
      ok = mbar_wait(bar_full(c), 0, abort_flag, err, kSiteKvFull, c);
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < kChunk / 16; ++kk)
        mma_ss(tD, ad0 + (uint64_t)((c * kChunkBytes + kk * 16 * 128) >> 4),
               bd0 + (uint64_t)((c * kChunkBytes + kk * 32) >> 4), kIdesc, (c | kk) != 0);
    }
    tc_commit(bar_done);  // arrives once every MMA issued above is complete
    if (!ok) {
      // let the copies this thread started land before the CTA unwinds
      for (int c = 0; c < nchunks; ++c) {
        volatile int never = 0;
        mbar_wait(bar_full(c), 0, &never, nullptr, kSiteDrain, c);
      }
    }
  }
  __syncwarp();

  // ---- epilogue: thread = output column m0 + threadIdx.x, 64 tokens each
  bool ok = mbar_wait(bar_done, 0, abort_flag, err, kSitePvDone, 0);
  ok = __all_sync(0xffffffffu, ok) && *abort_flag == 0;
  if (ok) {
    tc_fence_after();
    const int m = m0 + threadIdx.x;
    const uint32_t lane_addr = tD + ((uint32_t)(warp * 32) << 16);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float v[32];
      tmem_ld32(lane_addr + half * 32, v);
      if (m < M) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int b = b0 + half * 32 + j;
          if (b < B) y[((size_t)b * Hq + h) * ldy + m] = __float2bfloat16_rn(v[j]);
        }
      }
    }
  }
  // the rotary part passes through (first column tile only)
  if (rope != nullptr && blockIdx.y == 0) {
    const int per_row = d_rope / 8;  // 16-byte pieces
    for (int i = threadIdx.x; i < kTileN * per_row; i += kThreads) {
      const int b = b0 + i / per_row, p = i % per_row;
      if (b < B)
        *reinterpret_cast<uint4*>(y + ((size_t)b * Hq + h) * ldy + rope_off + p * 8) =
            *reinterpret_cast<const uint4*>(rope + ((size_t)b * Hq + h) * d_rope + p * 8);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tD, kTileN);
  }
}

// 3-D tensor map of bf16 elements with the 128-byte swizzle: dims and byte
// strides of the two outer dimensions, box {64, box1, box2}.
CUresult make_map(CUtensorMap* map, const void* ptr, cuuint64_t d0, cuuint64_t d1,
                  cuuint64_t d2, cuuint64_t s1, cuuint64_t s2, cuuint32_t box1,
                  cuuint32_t box2) {
  PFN_encodeTiled enc = get_encode_tiled();
  if (!enc) return CUDA_ERROR_NOT_FOUND;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {s1, s2};
  cuuint32_t box[3] = {64, box1, box2};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int fail(int code, const char* what, const char* why) {
  attn_set_error("%s: %s", what, why);
  return code;
}

// Y[b, h, 0:M] (row stride ldy) = X[b, h, 0:K] W[h, 0:K, 0:M] for every token
// b < B and head h; optionally rope[b, h, :] copied to Y[b, h, rope_off:].
int launch_proj(const char* what, const void* x, const void* w, void* y, int ldy,
                const void* rope, int d_rope, int rope_off, int B, int Hq, int K, int M,
                cudaStream_t s) {
  int code = ATTN_OK;
  int* err = attn_device_err_word(&code);
  if (!err) return code;
  CUtensorMap mw, mx;
  CUresult r = make_map(&mw, w, (cuuint64_t)M, (cuuint64_t)K, (cuuint64_t)Hq,
                        (cuuint64_t)M * 2, (cuuint64_t)K * M * 2, kChunk, 1);
  if (r == CUDA_SUCCESS)
    r = make_map(&mx, x, (cuuint64_t)K, (cuuint64_t)Hq, (cuuint64_t)B, (cuuint64_t)K * 2,
                 (cuuint64_t)Hq * K * 2, 1, kTileN);
  if (r != CUDA_SUCCESS) {
    attn_set_error("%s: cuTensorMapEncodeTiled failed (CUresult %d)", what, (int)r);
    return ATTN_ERR_CUDA;
  }
  cudaError_t e = cudaFuncSetAttribute(
      mla_proj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes(kMaxK));
  if (e == cudaSuccess) {
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(Hq, (M + kTileM - 1) / kTileM, (B + kTileN - 1) / kTileN);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem_bytes(K);
    cfg.stream = s;
    cfg.attrs = pdl;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, mla_proj_kernel, mw, mx, static_cast<__nv_bfloat16*>(y), ldy,
                           static_cast<const __nv_bfloat16*>(rope), d_rope, rope_off, B, Hq, K,
                           M, err);
  }
  if (e != cudaSuccess) {
    attn_set_error("%s: launch failed: %s", what, cudaGetErrorString(e));
    return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}

}  // namespace

extern "C" int mla_absorb_q(const void* q_nope, const void* q_rope, const void* w_uk,
                            void* q_out, int B, int Hq, int d_nope, int d_rope, int d_latent,
                            void* stream) {
  const char* what = "mla_absorb_q";
  attn_set_error("%s", "");
  if (!q_nope || !q_rope || !w_uk || !q_out)
    return fail(ATTN_ERR_INVALID_ARG, what, "null pointer argument");
  if (B <= 0 || Hq <= 0 || d_nope <= 0 || d_rope <= 0 || d_latent <= 0)
    return fail(ATTN_ERR_INVALID_ARG, what, "B, Hq and every width must be >= 1");
  if (d_nope % 8 || d_rope % 8 || d_latent % 8)
    return fail(ATTN_ERR_INVALID_ARG, what, "widths must be multiples of 8");
  if (d_nope % kChunk || d_nope > kMaxK || d_latent % 64)
    return fail(ATTN_ERR_UNSUPPORTED, what,
                "built for d_nope a multiple of 64 up to 512 and d_latent a multiple of 64");
  if ((long long)B * Hq * (d_latent + d_rope) > 0x7fffffffLL || Hq > 65535 ||
      B > 65535 * kTileN)
    return fail(ATTN_ERR_INVALID_ARG, what, "problem too large");
  if (!aligned16(q_nope) || !aligned16(q_rope) || !aligned16(w_uk) || !aligned16(q_out))
    return fail(ATTN_ERR_MISALIGNED, what, "pointers must be 16-byte aligned");
  return launch_proj(what, q_nope, w_uk, q_out, d_latent + d_rope, q_rope, d_rope, d_latent, B,
                     Hq, d_nope, d_latent, static_cast<cudaStream_t>(stream));
}

extern "C" int mla_project_out(const void* o_latent, const void* w_uv, void* out, int B, int Hq,
                               int d_latent, int d_v, void* stream) {
  const char* what = "mla_project_out";
  attn_set_error("%s", "");
  if (!o_latent || !w_uv || !out) return fail(ATTN_ERR_INVALID_ARG, what, "null pointer argument");
  if (B <= 0 || Hq <= 0 || d_latent <= 0 || d_v <= 0)
    return fail(ATTN_ERR_INVALID_ARG, what, "B, Hq and every width must be >= 1");
  if (d_latent % 8 || d_v % 8)
    return fail(ATTN_ERR_INVALID_ARG, what, "widths must be multiples of 8");
  if (d_latent % kChunk || d_latent > kMaxK || d_v % 64)
    return fail(ATTN_ERR_UNSUPPORTED, what,
                "built for d_latent a multiple of 64 up to 512 and d_v a multiple of 64");
  if ((long long)B * Hq * d_latent > 0x7fffffffLL || Hq > 65535 || B > 65535 * kTileN)
    return fail(ATTN_ERR_INVALID_ARG, what, "problem too large");
  if (!aligned16(o_latent) || !aligned16(w_uv) || !aligned16(out))
    return fail(ATTN_ERR_MISALIGNED, what, "pointers must be 16-byte aligned");
  return launch_proj(what, o_latent, w_uv, out, d_v, nullptr, 0, 0, B, Hq, d_latent, d_v,
                     static_cast<cudaStream_t>(stream));
}
