// attn_api.cu -- the extern "C" boundary of libattn.so (declared in
// include/attn.h): argument validation, the per-device error word, the
// tensor-map encoder entry point, and dispatch to the kernel launchers.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "common.cuh"

// ---------------------------------------------------------------- errors

static thread_local char g_msg[512] = "";

void attn_set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
}

extern "C" const char* attn_last_error(void) { return g_msg; }

static int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return code;
}

// One error word per device (a __device__ variable exists once per device
// context).  Its device address is looked up once per device.
__device__ int g_attn_err[gb300::kErrWords];

static constexpr int kMaxDevices = 64;
static int* g_err_ptr[kMaxDevices] = {};
static std::mutex g_err_mu;

static int* device_err_word(int* code_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *code_out = fail(ATTN_ERR_CUDA, "cudaGetDevice failed: %s", cudaGetErrorString(e));
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_err_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attn_err);
    if (e != cudaSuccess) {
      *code_out =
          fail(ATTN_ERR_CUDA, "cudaGetSymbolAddress(error word) failed: %s",
               cudaGetErrorString(e));
      return nullptr;
    }
    g_err_ptr[dev] = static_cast<int*>(p);
  }
  return g_err_ptr[dev];
}

int* attn_device_err_word(int* code_out) { return device_err_word(code_out); }

static int sm_count(int* code_out) {
  int dev = 0, n = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) {
    *code_out = fail(ATTN_ERR_CUDA, "device query failed: %s", cudaGetErrorString(e));
    return 0;
  }
  return n;
}

// ------------------------------------------------- tensor-map encoder entry

PFN_encodeTiled get_encode_tiled() {
  static PFN_encodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_encodeTiled>(p);
  });
  return fn;
}

// ---------------------------------------------------------------- helpers

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static int finish_launch(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return ATTN_OK;
  if (g_msg[0] == '\0' || e != cudaErrorInvalidValue)
    return fail(ATTN_ERR_CUDA, "%s: launch failed: %s", what, cudaGetErrorString(e));
  return ATTN_ERR_CUDA;
}

// ---------------------------------------------------------------- attn_fwd

static int attn_fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse,
                         int B, int H, int N, int D, int causal, float scale, int dtype,
                         void* stream, int debug_skip_load) {
  g_msg[0] = '\0';
  if (!q || !k || !v || !o || !lse)
    return fail(ATTN_ERR_INVALID_ARG, "attn_fwd: null pointer argument");
  if (B <= 0 || H <= 0 || N <= 0 || D <= 0)
    return fail(ATTN_ERR_INVALID_ARG, "attn_fwd: B, H, N, D must be >= 1 (got %d %d %d %d)",
                B, H, N, D);
  if (!isfinite(scale)) return fail(ATTN_ERR_INVALID_ARG, "attn_fwd: scale is not finite");
  if ((long long)B * H > 0x7fffffffLL)
    return fail(ATTN_ERR_INVALID_ARG, "attn_fwd: B*H too large");
  if (dtype == ATTN_DTYPE_F32) {
    if (D != 64) return fail(ATTN_ERR_UNSUPPORTED, "attn_fwd: fp32 path is built for D=64");
  } else if (dtype == ATTN_DTYPE_BF16) {
    if (D != 64 && D != 128)
      return fail(ATTN_ERR_UNSUPPORTED, "attn_fwd: bf16 path is built for D=64 and D=128");
    if ((long long)B * H * N > 0x7fffffffLL)
      return fail(ATTN_ERR_UNSUPPORTED, "attn_fwd: B*H*N exceeds the tensor-map range");
  } else {
    return fail(ATTN_ERR_UNSUPPORTED, "attn_fwd: unknown dtype %d", dtype);
  }
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return fail(ATTN_ERR_MISALIGNED, "attn_fwd: pointers must be 16-byte aligned");

  int code = ATTN_OK;
  int* err = device_err_word(&code);
  if (!err) return code;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == ATTN_DTYPE_F32) {
    // the fp32 hook passes its K/V block index plus one (0: none)
    PrefillF32Args a{static_cast<const float*>(q), static_cast<const float*>(k),
                     static_cast<const float*>(v), static_cast<float*>(o), lse, B, H, N, D,
                     causal != 0, scale, err, debug_skip_load - 1};
    return finish_launch(launch_prefill_f32(a, s), "attn_fwd");
  }
  int nsm = sm_count(&code);
  if (nsm <= 0) return code;
  PrefillBf16Args a{q, k, v, o, lse, B, H, N, D, causal != 0, scale, err, nsm,
                    debug_skip_load};
  return finish_launch(launch_prefill_bf16(a, s), "attn_fwd");
}

extern "C" int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                        int B, int H, int N, int D, int causal, float scale, int dtype,
                        void* stream) {
  return attn_fwd_impl(q, k, v, o, lse, B, H, N, D, causal, scale, dtype, stream, 0);
}

extern "C" int attn_fwd_f32_test_skip_load(const float* q, const float* k, const float* v,
                                           float* o, float* lse, int B, int H, int N, int D,
                                           int causal, float scale, void* stream,
                                           int skip_block) {
  if (skip_block < 0)
    return fail(ATTN_ERR_INVALID_ARG, "attn_fwd_f32_test_skip_load: block must be >= 0");
  return attn_fwd_impl(q, k, v, o, lse, B, H, N, D, causal, scale, ATTN_DTYPE_F32, stream,
                       skip_block + 1);
}

extern "C" int attn_fwd_test_skip_load(const void* q, const void* k, const void* v, void* o,
                                       float* lse, int B, int H, int N, int D, int causal,
                                       float scale, void* stream, int skip_load_index) {
  if (skip_load_index <= 0)
    return fail(ATTN_ERR_INVALID_ARG, "attn_fwd_test_skip_load: index must be >= 1");
  return attn_fwd_impl(q, k, v, o, lse, B, H, N, D, causal, scale, ATTN_DTYPE_BF16, stream,
                       skip_load_index);
}

// ------------------------------------------------------- attn_fwd_tf32x3

extern "C" size_t attn_fwd_tf32x3_workspace_size(int B, int H, int N, int D) {
  if (B <= 0 || H <= 0 || N <= 0 || D != 64) return 0;
  return prefill_tf32x3_workspace_bytes(B, H, N);
}

static int tf32x3_impl(const float* q, const float* k, const float* v, float* o, float* lse,
                       int B, int H, int N, int D, int causal, float scale, void* workspace,
                       size_t workspace_bytes, void* stream, int debug_skip_block) {
  g_msg[0] = '\0';
  if (!q || !k || !v || !o || !lse || !workspace)
    return fail(ATTN_ERR_INVALID_ARG, "attn_fwd_tf32x3: null pointer argument");
  if (B <= 0 || H <= 0 || N <= 0 || D <= 0)
    return fail(ATTN_ERR_INVALID_ARG,
                "attn_fwd_tf32x3: B, H, N, D must be >= 1 (got %d %d %d %d)", B, H, N, D);
  if (!isfinite(scale))
    return fail(ATTN_ERR_INVALID_ARG, "attn_fwd_tf32x3: scale is not finite");
  if (D != 64) return fail(ATTN_ERR_UNSUPPORTED, "attn_fwd_tf32x3: built for D=64 (got %d)", D);
  if ((long long)B * H * N > 0x7fffffffLL)
    return fail(ATTN_ERR_UNSUPPORTED, "attn_fwd_tf32x3: B*H*N exceeds the tensor-map range");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(workspace))
    return fail(ATTN_ERR_MISALIGNED, "attn_fwd_tf32x3: pointers must be 16-byte aligned");
  const size_t need = prefill_tf32x3_workspace_bytes(B, H, N);
  if (workspace_bytes < need)
    return fail(ATTN_ERR_WORKSPACE_TOO_SMALL, "attn_fwd_tf32x3: workspace %zu < %zu bytes",
                workspace_bytes, need);
  int code = ATTN_OK;
  int* err = device_err_word(&code);
  if (!err) return code;
  PrefillTf32x3Args a{q, k, v, o, lse, B, H, N, D, causal != 0, scale, workspace, err,
                      debug_skip_block};
  return finish_launch(launch_prefill_tf32x3(a, static_cast<cudaStream_t>(stream)),
                       "attn_fwd_tf32x3");
}

extern "C" int attn_fwd_tf32x3(const float* q, const float* k, const float* v, float* o,
                               float* lse, int B, int H, int N, int D, int causal, float scale,
                               void* workspace, size_t workspace_bytes, void* stream) {
  return tf32x3_impl(q, k, v, o, lse, B, H, N, D, causal, scale, workspace, workspace_bytes,
                     stream, -1);
}

extern "C" int attn_fwd_tf32x3_test_skip_load(const float* q, const float* k, const float* v,
                                              float* o, float* lse, int B, int H, int N, int D,
                                              int causal, float scale, void* workspace,
                                              size_t workspace_bytes, void* stream,
                                              int skip_block) {
  if (skip_block < 0)
    return fail(ATTN_ERR_INVALID_ARG, "attn_fwd_tf32x3_test_skip_load: block must be >= 0");
  return tf32x3_impl(q, k, v, o, lse, B, H, N, D, causal, scale, workspace, workspace_bytes,
                     stream, skip_block);
}

// ---------------------------------------------------------------- MLA

extern "C" size_t mla_decode_split_workspace_size(int B, int Hq, int max_blocks_per_seq,
                                                  int num_sms, int pages_per_split) {
  if (B <= 0 || Hq <= 0 || max_blocks_per_seq <= 0 || num_sms < 2 || pages_per_split < 0)
    return 0;
  return mla_workspace_bytes(B, Hq, max_blocks_per_seq, num_sms, pages_per_split);
}

extern "C" size_t mla_decode_workspace_size(int B, int Hq, int max_blocks_per_seq,
                                            int num_sms) {
  return mla_decode_split_workspace_size(B, Hq, max_blocks_per_seq, num_sms, 0);
}

static int mla_impl(const void* q, const void* kv, const int32_t* table, const int32_t* seqlens,
                    void* o, float* lse, int B, int Hq, float scale, int max_blocks,
                    int num_blocks, void* ws, size_t ws_bytes, int pages_per_split,
                    void* stream, int debug_skip_step = -1) {
  g_msg[0] = '\0';
  if (!q || !kv || !table || !seqlens || !o || !lse || !ws)
    return fail(ATTN_ERR_INVALID_ARG, "mla_decode: null pointer argument");
  if (B <= 0 || Hq <= 0 || max_blocks <= 0 || num_blocks <= 0 || pages_per_split < 0)
    return fail(ATTN_ERR_INVALID_ARG, "mla_decode: sizes must be >= 1");
  if (!isfinite(scale)) return fail(ATTN_ERR_INVALID_ARG, "mla_decode: scale is not finite");
  if (Hq != 128) return fail(ATTN_ERR_UNSUPPORTED, "mla_decode: built for Hq=128 (got %d)", Hq);
  if ((long long)num_blocks * 64 > 0x7fffffffLL || (long long)B * max_blocks > 0x7fffffffLL)
    return fail(ATTN_ERR_UNSUPPORTED, "mla_decode: pool or table too large");
  if (!aligned16(q) || !aligned16(kv) || !aligned16(o) || !aligned16(lse) || !aligned16(ws) ||
      !aligned16(table) || !aligned16(seqlens))
    return fail(ATTN_ERR_MISALIGNED, "mla_decode: pointers must be 16-byte aligned");
  int code = ATTN_OK;
  const int nsm = sm_count(&code);
  if (nsm <= 0) return code;
  const size_t need = mla_workspace_bytes(B, Hq, max_blocks, nsm, pages_per_split);
  if (ws_bytes < need)
    return fail(ATTN_ERR_WORKSPACE_TOO_SMALL, "mla_decode: workspace %zu < %zu bytes",
                ws_bytes, need);
  int* err = device_err_word(&code);
  if (!err) return code;
  MlaArgs a{q, kv, table, seqlens, o, lse, B, Hq, scale, max_blocks, num_blocks, ws, ws_bytes,
            pages_per_split, nsm, err, debug_skip_step};
  return finish_launch(launch_mla_decode(a, static_cast<cudaStream_t>(stream)), "mla_decode");
}

extern "C" int mla_decode(const void* q, const void* kv_cache, const int32_t* block_table,
                          const int32_t* seqlens, void* o, float* lse, int B, int Hq,
                          float scale, int max_blocks_per_seq, int num_blocks, void* workspace,
                          size_t workspace_bytes, void* stream) {
  return mla_impl(q, kv_cache, block_table, seqlens, o, lse, B, Hq, scale, max_blocks_per_seq,
                  num_blocks, workspace, workspace_bytes, 0, stream);
}

extern "C" int mla_decode_split(const void* q, const void* kv_cache,
                                const int32_t* block_table, const int32_t* seqlens, void* o,
                                float* lse, int B, int Hq, float scale, int max_blocks_per_seq,
                                int num_blocks, void* workspace, size_t workspace_bytes,
                                int pages_per_split, void* stream) {
  return mla_impl(q, kv_cache, block_table, seqlens, o, lse, B, Hq, scale, max_blocks_per_seq,
                  num_blocks, workspace, workspace_bytes, pages_per_split, stream);
}

extern "C" int mla_decode_test_skip_load(const void* q, const void* kv_cache,
                                         const int32_t* block_table, const int32_t* seqlens,
                                         void* o, float* lse, int B, int Hq, float scale,
                                         int max_blocks_per_seq, int num_blocks,
                                         void* workspace, size_t workspace_bytes,
                                         void* stream, int skip_step) {
  if (skip_step < 0)
    return fail(ATTN_ERR_INVALID_ARG, "mla_decode_test_skip_load: step must be >= 0");
  return mla_impl(q, kv_cache, block_table, seqlens, o, lse, B, Hq, scale, max_blocks_per_seq,
                  num_blocks, workspace, workspace_bytes, 0, stream, skip_step);
}

extern "C" int mla_decode_noalloc(const void* q, const void* kv_cache,
                                  const int32_t* block_table, const int32_t* seqlens,
                                  void* o, float* lse, int B, int Hq, float scale,
                                  int max_blocks_per_seq, int num_blocks, void* stream) {
  g_msg[0] = '\0';
  if (B > mla_noalloc_max_batch())
    return fail(ATTN_ERR_UNSUPPORTED,
                "mla_decode_noalloc: B=%d exceeds the fixed-scratch limit of %d sequences", B,
                mla_noalloc_max_batch());
  int code = ATTN_OK;
  const int nsm = sm_count(&code);
  if (nsm <= 0) return code;
  if (nsm > mla_noalloc_max_sms())
    return fail(ATTN_ERR_UNSUPPORTED,
                "mla_decode_noalloc: device has %d SMs, the fixed scratch covers %d", nsm,
                mla_noalloc_max_sms());
  void* ws = nullptr;
  size_t ws_bytes = 0;
  cudaError_t e = mla_noalloc_scratch(&ws, &ws_bytes);
  if (e != cudaSuccess)
    return fail(ATTN_ERR_CUDA, "mla_decode_noalloc: cudaGetSymbolAddress failed: %s",
                cudaGetErrorString(e));
  return mla_impl(q, kv_cache, block_table, seqlens, o, lse, B, Hq, scale, max_blocks_per_seq,
                  num_blocks, ws, ws_bytes, 0, stream);
}

// ---------------------------------------------------------------- status

extern "C" int attn_device_status(void* stream) {
  g_msg[0] = '\0';
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess)
    return fail(ATTN_ERR_CUDA, "attn_device_status: stream error: %s", cudaGetErrorString(e));
  int code = ATTN_OK;
  int* err = device_err_word(&code);
  if (!err) return code;
  int h[gb300::kErrWords] = {0, 0, 0, 0};
  e = cudaMemcpy(h, err, sizeof(h), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess)
    return fail(ATTN_ERR_CUDA, "attn_device_status: read failed: %s", cudaGetErrorString(e));
  if (h[0] == 0) return ATTN_OK;
  const int zero[gb300::kErrWords] = {0, 0, 0, 0};
  e = cudaMemcpy(err, zero, sizeof(zero), cudaMemcpyHostToDevice);
  if (e != cudaSuccess)
    return fail(ATTN_ERR_CUDA, "attn_device_status: clear failed: %s", cudaGetErrorString(e));
  const char* what = h[0] == ATTN_ERR_DEVICE_TIMEOUT   ? "pipeline wait ran out"
                     : h[0] == ATTN_ERR_BAD_BLOCK_TABLE ? "block-table entry out of range"
                     : h[0] == ATTN_ERR_BAD_SEQLEN      ? "sequence length out of range"
                                                        : "device error";
  return fail(h[0], "device: %s (site %d, block %d, detail %d)", what, h[1], h[2], h[3]);
}

// ---------------------------------------------------------------- helpers

extern "C" int attn_kv_tiles(int N, int Br, int Bc, int causal, int q_tile) {
  if (N <= 0 || Br <= 0 || Bc <= 0 || q_tile < 0 || (long long)q_tile * Br >= N) return -1;
  const long long q_start = (long long)q_tile * Br;
  const long long kv_limit = causal ? (q_start + Br < N ? q_start + Br : N) : N;
  return (int)((kv_limit + Bc - 1) / Bc);
}

extern "C" int attn_kernel_info(int dtype, int D, int* Br, int* Bc, int* threads,
                                int* smem_bytes) {
  bool ok = false;
  if (dtype == ATTN_DTYPE_F32) ok = prefill_f32_info(D, Br, Bc, threads, smem_bytes);
  else if (dtype == ATTN_DTYPE_BF16) ok = prefill_bf16_info(D, Br, Bc, threads, smem_bytes);
  return ok ? ATTN_OK : fail(ATTN_ERR_UNSUPPORTED, "attn_kernel_info: not built");
}
