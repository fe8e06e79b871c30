// mla_absorb.cu -- the two projections around MLA absorbed decode.
//
// The "MLA x FlashAttention-3 fusion" article (hnwysp news 119127) folds the
// per-head up-projections into the query and the output: with the latent
// row c_t (512) and per-head W_UK, W_UV, the score of head h is
//   q_nope_h . (W_UK_h^T c_t) + q_rope_h . k_rope_t = (q_nope_h W_UK_h) . c_t + ...
// (the absorption identity), and its output is (sum_t p_t c_t) W_UV_h.  So
// the decode kernel needs the absorbed query [q_nope_h W_UK_h | q_rope_h]
// (576 wide) and leaves a 512-wide latent output that W_UV_h maps to the
// head's values.  Both are plain per-head GEMMs (a batch of Hq independent
// matrix products); they run as cuBLAS strided-batched GEMMs, bf16 operands
// with fp32 accumulation, on the caller's stream.
#include <cublas_v2.h>

#include <mutex>

#include "common.cuh"

namespace {

// One cuBLAS handle per device, created on first use and bound to the
// caller's stream for each call under a lock.
constexpr int kMaxDevs = 64;
cublasHandle_t g_handle[kMaxDevs] = {};
std::mutex g_mu;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int fail_args(const char* what, const char* why) {
  attn_set_error("%s: %s", what, why);
  return ATTN_ERR_INVALID_ARG;
}

// Runs C_h = A_h . W_h for every head h (row-major, bf16): A_h is row b of
// [B][Hq][k] at head h, W_h is [k][n] contiguous per head, C_h goes to row b
// of [B][Hq][ldc_row] at head h (first n entries).  In cuBLAS's column-major
// terms this is C_h^T (n x B) = W_h^T (n x k) . A_h^T (k x B).
int batched_rows_times_weights(const char* what, const void* a, const void* w, void* c, int B,
                               int Hq, int k, int n, int ldc_row, cudaStream_t s) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevs) {
    attn_set_error("%s: no usable CUDA device", what);
    return ATTN_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_handle[dev] == nullptr) {
    const cublasStatus_t st = cublasCreate(&g_handle[dev]);
    if (st != CUBLAS_STATUS_SUCCESS) {
      g_handle[dev] = nullptr;
      attn_set_error("%s: cublasCreate failed (status %d)", what, (int)st);
      return ATTN_ERR_CUDA;
    }
  }
  cublasHandle_t h = g_handle[dev];
  cublasStatus_t st = cublasSetStream(h, s);
  if (st == CUBLAS_STATUS_SUCCESS) {
    const float alpha = 1.f, beta = 0.f;
    st = cublasGemmStridedBatchedEx(h, CUBLAS_OP_N, CUBLAS_OP_N, n, B, k, &alpha,
                                    w, CUDA_R_16BF, n, (long long)k * n,
                                    a, CUDA_R_16BF, Hq * k, k, &beta,
                                    c, CUDA_R_16BF, Hq * ldc_row, ldc_row, Hq,
                                    CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
  }
  if (st != CUBLAS_STATUS_SUCCESS) {
    attn_set_error("%s: cuBLAS GEMM failed (status %d)", what, (int)st);
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
  if (!q_nope || !q_rope || !w_uk || !q_out) return fail_args(what, "null pointer argument");
  if (B <= 0 || Hq <= 0 || d_nope <= 0 || d_rope <= 0 || d_latent <= 0)
    return fail_args(what, "B, Hq and every width must be >= 1");
  if (d_nope % 8 || d_rope % 8 || d_latent % 8)
    return fail_args(what, "widths must be multiples of 8 (16-byte bf16 rows)");
  if ((long long)B * Hq * (d_latent + d_rope) > 0x7fffffffLL ||
      (long long)Hq * (d_latent + d_rope) > 0x7fffffffLL)
    return fail_args(what, "problem too large");
  if (!aligned16(q_nope) || !aligned16(q_rope) || !aligned16(w_uk) || !aligned16(q_out)) {
    attn_set_error("%s: pointers must be 16-byte aligned", what);
    return ATTN_ERR_MISALIGNED;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int row = d_latent + d_rope;
  const int code =
      batched_rows_times_weights(what, q_nope, w_uk, q_out, B, Hq, d_nope, d_latent, row, s);
  if (code != ATTN_OK) return code;
  // q_rope passes through into the last d_rope entries of each row
  const cudaError_t e = cudaMemcpy2DAsync(
      static_cast<__nv_bfloat16*>(q_out) + d_latent, (size_t)row * 2, q_rope, (size_t)d_rope * 2,
      (size_t)d_rope * 2, (size_t)B * Hq, cudaMemcpyDeviceToDevice, s);
  if (e != cudaSuccess) {
    attn_set_error("%s: copy of q_rope failed: %s", what, cudaGetErrorString(e));
    return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}

extern "C" int mla_project_out(const void* o_latent, const void* w_uv, void* out, int B, int Hq,
                               int d_latent, int d_v, void* stream) {
  const char* what = "mla_project_out";
  attn_set_error("%s", "");
  if (!o_latent || !w_uv || !out) return fail_args(what, "null pointer argument");
  if (B <= 0 || Hq <= 0 || d_latent <= 0 || d_v <= 0)
    return fail_args(what, "B, Hq and every width must be >= 1");
  if (d_latent % 8 || d_v % 8) return fail_args(what, "widths must be multiples of 8");
  if ((long long)B * Hq * d_latent > 0x7fffffffLL || (long long)Hq * d_latent > 0x7fffffffLL ||
      (long long)B * Hq * d_v > 0x7fffffffLL)
    return fail_args(what, "problem too large");
  if (!aligned16(o_latent) || !aligned16(w_uv) || !aligned16(out)) {
    attn_set_error("%s: pointers must be 16-byte aligned", what);
    return ATTN_ERR_MISALIGNED;
  }
  return batched_rows_times_weights(what, o_latent, w_uv, out, B, Hq, d_latent, d_v, d_v,
                                    static_cast<cudaStream_t>(stream));
}
